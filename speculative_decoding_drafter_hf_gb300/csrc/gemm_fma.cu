// CUDA-core GEMM with fused epilogues: Y[r, c] = sum_k X[r, k] * Wt[c, k].
//
// Used for the fp32 mode, where the tensor pipe's tf32 rounding (10-bit
// mantissa) would break the 1e-4 parity bar. Operands are staged through
// shared memory as fp32; accumulation is fp32. Split-K partials are summed in
// a fixed order by a second kernel, so results are deterministic.
#include "common.cuh"

namespace hf {
namespace {

constexpr int BM = 64, BN = 64, BK = 32;

template <typename T>
__global__ void __launch_bounds__(256)
gemm_fma_kernel(const T* __restrict__ X, int ldx, const T* __restrict__ Wt, int ldw, int R,
                int C, int K, int kchunk, float* __restrict__ part, Epi epi) {
  __shared__ __align__(16) float As[BK][BM + 4];
  __shared__ __align__(16) float Bs[BK][BN + 4];
  const int r0 = blockIdx.y * BM, c0 = blockIdx.x * BN;
  const int kb = blockIdx.z * kchunk;
  const int ke = min(K, kb + kchunk);
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = kb; k0 < ke; k0 += BK) {
    for (int i = tid; i < BM * BK; i += 256) {
      int rr = i / BK, kk = i % BK, r = r0 + rr, k = k0 + kk;
      As[kk][rr] = (r < R && k < ke) ? to_f(X[(size_t)r * ldx + k]) : 0.f;
    }
    for (int i = tid; i < BN * BK; i += 256) {
      int cc = i / BK, kk = i % BK, c = c0 + cc, k = k0 + kk;
      Bs[kk][cc] = (c < C && k < ke) ? to_f(Wt[(size_t)c * ldw + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int r = r0 + ty * 4 + i;
    if (r >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int c = c0 + tx * 4 + j;
      if (c >= C) continue;
      if (gridDim.z == 1)
        epi_apply<T>(epi, r, c, acc[i][j]);
      else
        part[((size_t)blockIdx.z * R + r) * C + c] = acc[i][j];
    }
  }
}

template <typename T>
__global__ void splitk_finish_kernel(const float* __restrict__ part, int splits, int R, int C,
                                     Epi epi) {
  const size_t n = (size_t)R * C;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < splits; ++s) v += part[(size_t)s * n + i];
    epi_apply<T>(epi, (int)(i / C), (int)(i % C), v);
  }
}

template <typename T>
cudaError_t run(const void* X, int ldx, const void* Wt, int ldw, int R, int C, int K, int splits,
                float* part, const Epi& epi, cudaStream_t st, int* launches) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (splits < 1) splits = 1;
  int kchunk = (K + splits - 1) / splits;
  kchunk = (kchunk + BK - 1) / BK * BK;
  splits = (K + kchunk - 1) / kchunk;
  dim3 grid((C + BN - 1) / BN, (R + BM - 1) / BM, splits);
  gemm_fma_kernel<T><<<grid, 256, 0, st>>>((const T*)X, ldx, (const T*)Wt, ldw, R, C, K, kchunk,
                                           part, epi);
  ++*launches;
  if (splits > 1) {
    size_t n = (size_t)R * C;
    int blocks = (int)std::min<size_t>((n + 255) / 256, 152 * 8);
    splitk_finish_kernel<T><<<blocks, 256, 0, st>>>(part, splits, R, C, epi);
    ++*launches;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_fma(int dtype, const void* X, int ldx, const void* Wt, int ldw, int R,
                            int C, int K, int splits, float* part, const Epi& epi,
                            cudaStream_t st, int* launches) {
  if (dtype == HF_F32)
    return run<float>(X, ldx, Wt, ldw, R, C, K, splits, part, epi, st, launches);
  return run<__nv_bfloat16>(X, ldx, Wt, ldw, R, C, K, splits, part, epi, st, launches);
}

}  // namespace hf
