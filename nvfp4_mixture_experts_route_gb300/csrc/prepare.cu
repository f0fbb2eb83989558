// moe_prepare_weights: raw NVFP4 experts -> the library's prepared layout
// (documented in include/moe_nvfp4.h). A one-time copy at load.
#include "common.cuh"
#include "layout.cuh"

namespace moe {

// p_w13[e, r, :] = w13[e, src(r), :] -- one 16-byte vector per thread step.
__global__ void __launch_bounds__(256) prepare_w13_kernel(const uint4* __restrict__ w13,
                                                          uint4* __restrict__ p_w13, int E, int I,
                                                          int row_vecs) {
  const long long total = (long long)E * 2 * I * row_vecs;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long row = idx / row_vecs;
    const int v = (int)(idx % row_vecs);
    const int e = (int)(row / (2 * I)), r = (int)(row % (2 * I));
    const long long src = ((long long)e * 2 * I + w13_source_row(r, I)) * row_vecs + v;
    p_w13[idx] = w13[src];
  }
}

// Scale atoms: each thread writes one 16-byte atom row (m0): the four 32-row
// groups m1 x the four blocks c of one k-atom.
__global__ void __launch_bounds__(256) prepare_sf_kernel(const uint8_t* __restrict__ sf,
                                                         uint8_t* __restrict__ atoms, int E,
                                                         int rows, int nb, int permute_w13,
                                                         int I) {
  const int kc = nb / 4;
  const long long total = (long long)E * (rows / kAtomRows) * kc * 32;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int m0 = (int)(idx % 32);
    const long long a = idx / 32;  // atom index (e, mt, k)
    const int k = (int)(a % kc);
    const long long em = a / kc;
    const int mt = (int)(em % (rows / kAtomRows));
    const int e = (int)(em / (rows / kAtomRows));
    uint32_t w[4];
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1) {
      const int r = mt * kAtomRows + 32 * m1 + m0;
      const int src = permute_w13 ? w13_source_row(r, I) : r;
      const uint8_t* s = sf + ((size_t)e * rows + src) * nb + 4 * k;
      w[m1] = (uint32_t)s[0] | ((uint32_t)s[1] << 8) | ((uint32_t)s[2] << 16) |
              ((uint32_t)s[3] << 24);
    }
    *reinterpret_cast<uint4*>(atoms + a * kAtomBytes + 16 * m0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

static int grid_for(long long work) {
  long long g = (work + 255) / 256;
  if (g < 1) g = 1;
  if (g > 152 * 32) g = 152 * 32;
  return (int)g;
}

cudaError_t launch_prepare_weights(const void* w13, const void* w13_sf, const void* w2,
                                   const void* w2_sf, int E, int H, int I, void* p_w13,
                                   void* p_w13_sf, void* p_w2, void* p_w2_sf,
                                   cudaStream_t stream) {
  const int row_vecs = (H / 2) / 16;
  prepare_w13_kernel<<<grid_for((long long)E * 2 * I * row_vecs), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(w13), reinterpret_cast<uint4*>(p_w13), E, I, row_vecs);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  prepare_sf_kernel<<<grid_for((long long)E * 2 * I / 4 * (H / 64)), 256, 0, stream>>>(
      reinterpret_cast<const uint8_t*>(w13_sf), reinterpret_cast<uint8_t*>(p_w13_sf), E, 2 * I,
      H / 16, 1, I);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  err = cudaMemcpyAsync(p_w2, w2, (size_t)E * H * (I / 2), cudaMemcpyDeviceToDevice, stream);
  if (err != cudaSuccess) return err;
  prepare_sf_kernel<<<grid_for((long long)E * H / 4 * (I / 64)), 256, 0, stream>>>(
      reinterpret_cast<const uint8_t*>(w2_sf), reinterpret_cast<uint8_t*>(p_w2_sf), E, H, I / 16,
      0, I);
  return cudaGetLastError();
}

}  // namespace moe
