// Index arithmetic of the library's layouts (prepared weights, workspace).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kAtomRows = 128;   // rows of one scale atom
constexpr int kAtomBytes = 512;  // 32 x 16 bytes

// Scale atoms per K=64 step of a route tile of tile_m rows (128 rows each).
__host__ __device__ __forceinline__ int sf_atoms_per_tile(int tile_m) {
  return (tile_m + kAtomRows - 1) / kAtomRows;
}

// Byte of scale (row r, 16-element block b) inside an atom.
__host__ __device__ __forceinline__ int atom_byte(int r, int b) {
  return 16 * (r & 31) + 4 * ((r & 127) >> 5) + (b & 3);
}

// Workspace activations / intermediate (the route operand of the GEMMs):
// scales of permuted row p (route tile tau = p / tile_m, row i in the tile)
// and 16-element block b, with kc = K/64 atoms along K and S atoms of 128
// rows per K=64 step: the atom of step b / 4 and rows [128 (i/128), +128) of
// the tile. Every K=64 MMA reads its scales from its own 4-column group of
// tensor memory, which one tcgen05.cp of such an atom fills.
__host__ __device__ __forceinline__ size_t act_sf_offset(int p, int b, int tile_m, int kc, int S) {
  const int tau = p / tile_m, i = p - tau * tile_m;
  return ((size_t)((size_t)tau * kc + (b >> 2)) * S + (i >> 7)) * kAtomBytes + atom_byte(i, b);
}

// Prepared weights: scales of (expert e, prepared row r, block b) for a
// tensor with `rows` rows per expert and kc = K/64 atoms along K.
__host__ __device__ __forceinline__ size_t weight_sf_offset(int e, int r, int b, int rows,
                                                            int kc) {
  return ((size_t)((size_t)e * (rows / kAtomRows) + (r >> 7)) * kc + (b >> 2)) * kAtomBytes +
         atom_byte(r, b);
}

// Raw w13 row feeding prepared row r (gate/up alternate in 16-row granules).
__host__ __device__ __forceinline__ int w13_source_row(int r, int I) {
  const int g = r >> 5, j = r & 31;
  return j < 16 ? 16 * g + j : I + 16 * g + (j - 16);
}

}  // namespace moe
