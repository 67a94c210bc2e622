// Prefill helpers: reset a request, fill its window from the last W prefix
// features, fold the prefix into its memory, set its position.
//
// Source: HyFlash abstract ("recurrent memory compresses historical target
// features into fixed-size states") and the explainer's "That is HyFlash":
// the memory holds the compressed history of committed target features.
// Folding a prefix is committing all of its features at once, from h = 0.
#include "common.cuh"

namespace hf {
namespace {

__global__ void prefill_reset_kernel(Dims d, const int32_t* __restrict__ reqs,
                                     float* __restrict__ state, int32_t* __restrict__ tags,
                                     int64_t* __restrict__ pos) {
  const int b = reqs[blockIdx.x];
  const size_t per = (size_t)d.Hm * d.P * d.N;
  for (int l = 0; l < d.L; ++l) {
    float4* h = reinterpret_cast<float4*>(state + ((size_t)l * d.Bmax + b) * per);
    for (size_t i = threadIdx.x; i < per / 4; i += blockDim.x) h[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i = threadIdx.x; i < d.W; i += blockDim.x) tags[(size_t)b * d.W + i] = -1;
  if (threadIdx.x == 0) pos[b] = 0;
}

// grid (n_rows): packed ring row j -> request i, its position, gathered row.
template <typename T>
__global__ void prefill_ring_prep_kernel(Dims d, int n_req, const int32_t* __restrict__ lens,
                                         const int32_t* __restrict__ reqs,
                                         const T* __restrict__ feats,
                                         int32_t* __restrict__ row_req,
                                         int64_t* __restrict__ row_pos,
                                         int32_t* __restrict__ tags, T* __restrict__ packed) {
  const int j = blockIdx.x;
  __shared__ long long s_src;
  __shared__ int s_found;
  if (threadIdx.x == 0) {
    long long cu = 0;
    int roff = 0;
    s_found = 0;
    for (int i = 0; i < n_req; ++i) {
      const int L = lens[i];
      const int nk = L < d.W ? L : d.W;
      if (j < roff + nk) {
        const int jj = j - roff;
        const long long p = (long long)L - nk + jj;
        const int b = reqs[i];
        row_req[j] = b;
        row_pos[j] = p;
        tags[(size_t)b * d.W + (int)(p % d.W)] = (int32_t)p;
        s_src = cu + p;
        s_found = 1;
        break;
      }
      roff += nk;
      cu += L;
    }
  }
  __syncthreads();
  if (!s_found) return;
  const T* src = feats + (size_t)s_src * d.D;
  T* dst = packed + (size_t)j * d.D;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) dst[i] = src[i];
}

// grid (Hm, n_req): token-by-token fold of the rows [seg0, seg1) of the packed
// prefix that belong to request i, starting from the state in memory.
constexpr int SCAN_TC = 32;   // tokens staged per step
constexpr int SCAN_QPT = 8;   // float4 state elements per thread (P*N <= 8192)

__global__ void __launch_bounds__(256)
prefill_scan_kernel(Dims d, int layer, const int32_t* __restrict__ lens,
                    const int32_t* __restrict__ reqs, long long seg0, long long seg1,
                    const float* __restrict__ xbd, const float* __restrict__ A_log,
                    float* __restrict__ state) {
  extern __shared__ __align__(16) float sm[];
  const int hd = blockIdx.x, i = blockIdx.y;
  long long cu = 0;
  for (int k = 0; k < i; ++k) cu += lens[k];
  const long long t0 = cu > seg0 ? cu : seg0;
  const long long tend = cu + lens[i];
  const long long t1 = tend < seg1 ? tend : seg1;
  if (t0 >= t1) return;
  const int b = reqs[i];
  const int P = d.P, N = d.N;
  const float A = -expf(A_log[layer * d.Hm + hd]);
  float4* h = reinterpret_cast<float4*>(state + ((((size_t)layer * d.Bmax + b) * d.Hm + hd) * P) * N);
  const int nq = P * N / 4;

  float4 hv[SCAN_QPT];
  int qp[SCAN_QPT], qn[SCAN_QPT];
#pragma unroll
  for (int u = 0; u < SCAN_QPT; ++u) {
    int q = threadIdx.x + u * blockDim.x;
    qp[u] = (q * 4) / N;
    qn[u] = (q * 4) % N;
    hv[u] = q < nq ? h[q] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float* xs = sm;                       // [TC][P]
  float* bs = xs + SCAN_TC * P;         // [TC][N]
  float* ds = bs + SCAN_TC * N;         // [TC]
  for (long long c0 = t0; c0 < t1; c0 += SCAN_TC) {
    const int nt = (int)((t1 - c0) < SCAN_TC ? (t1 - c0) : SCAN_TC);
    __syncthreads();
    for (int k = threadIdx.x; k < nt * P; k += blockDim.x) {
      int t = k / P, p = k % P;
      xs[t * P + p] = xbd[(size_t)(c0 - seg0 + t) * d.NS + hd * P + p];
    }
    for (int k = threadIdx.x; k < nt * N; k += blockDim.x) {
      int t = k / N, n = k % N;
      bs[t * N + n] = xbd[(size_t)(c0 - seg0 + t) * d.NS + d.dinner + n];
    }
    for (int k = threadIdx.x; k < nt; k += blockDim.x)
      ds[k] = xbd[(size_t)(c0 - seg0 + k) * d.NS + d.dinner + d.N + hd];
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
      const float dt = ds[t];
      const float dec = expf(dt * A);
#pragma unroll
      for (int u = 0; u < SCAN_QPT; ++u) {
        int q = threadIdx.x + u * blockDim.x;
        if (q < nq) {
          const float xv = dt * xs[t * P + qp[u]];
          const float4 Bv = *reinterpret_cast<const float4*>(&bs[t * N + qn[u]]);
          hv[u].x = fmaf(dec, hv[u].x, xv * Bv.x);
          hv[u].y = fmaf(dec, hv[u].y, xv * Bv.y);
          hv[u].z = fmaf(dec, hv[u].z, xv * Bv.z);
          hv[u].w = fmaf(dec, hv[u].w, xv * Bv.w);
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < SCAN_QPT; ++u) {
    int q = threadIdx.x + u * blockDim.x;
    if (q < nq) h[q] = hv[u];
  }
}

__global__ void prefill_finish_kernel(int n_req, const int32_t* __restrict__ lens,
                                      const int32_t* __restrict__ reqs, int64_t* __restrict__ pos) {
  for (int i = threadIdx.x + blockIdx.x * blockDim.x; i < n_req; i += blockDim.x * gridDim.x)
    pos[reqs[i]] = lens[i];
}

}  // namespace

cudaError_t launch_prefill_reset(const Dims& d, int n_req, const int32_t* reqs, float* state,
                                 int32_t* tags, int64_t* pos, cudaStream_t st) {
  if (n_req <= 0) return cudaSuccess;
  prefill_reset_kernel<<<n_req, 256, 0, st>>>(d, reqs, state, tags, pos);
  return cudaGetLastError();
}

cudaError_t launch_prefill_ring_prep(int dtype, const Dims& d, int n_req, int n_rows,
                                     const int32_t* lens, const int32_t* reqs, const void* feats,
                                     int32_t* row_req, int64_t* row_pos, int32_t* tags,
                                     void* packed, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (dtype == HF_F32)
    prefill_ring_prep_kernel<float><<<n_rows, 128, 0, st>>>(
        d, n_req, lens, reqs, (const float*)feats, row_req, row_pos, tags, (float*)packed);
  else
    prefill_ring_prep_kernel<__nv_bfloat16><<<n_rows, 128, 0, st>>>(
        d, n_req, lens, reqs, (const __nv_bfloat16*)feats, row_req, row_pos, tags,
        (__nv_bfloat16*)packed);
  return cudaGetLastError();
}

cudaError_t launch_prefill_scan(const Dims& d, int layer, int n_req, const int32_t* lens,
                                const int32_t* reqs, long long seg0, long long seg1,
                                const float* xbd, const float* A_log, float* state,
                                cudaStream_t st) {
  if (n_req <= 0 || seg1 <= seg0) return cudaSuccess;
  size_t smem = (size_t)SCAN_TC * (d.P + d.N + 1) * sizeof(float);
  prefill_scan_kernel<<<dim3(d.Hm, n_req), 256, smem, st>>>(d, layer, lens, reqs, seg0, seg1, xbd,
                                                            A_log, state);
  return cudaGetLastError();
}

cudaError_t launch_prefill_finish(int n_req, const int32_t* lens, const int32_t* reqs,
                                  int64_t* pos, cudaStream_t st) {
  if (n_req <= 0) return cudaSuccess;
  prefill_finish_kernel<<<1, 256, 0, st>>>(n_req, lens, reqs, pos);
  return cudaGetLastError();
}

}  // namespace hf
