// Commit path: accepted-count check, packed row offsets, ring positions,
// and the sequential memory update.
//
// Source: learnaivisually explainer, FAQ "Why does the memory update only
// from committed features?" and "That is HyFlash": after verification only
// the newly committed features update the state, in order; drafting never
// writes it. Ring slots follow the sliding-window rule (Jargon,
// "Sliding-window attention"): the window keeps the most recent W committed
// positions, position t in slot t mod W.
#include "common.cuh"

namespace hf {
namespace {

constexpr int QPT = 2;  // float4 state elements per thread of the state update

// grid (B, S+1): CTA (b, t) owns accepted row t of request b.
template <typename T>
__global__ void __launch_bounds__(128)
commit_prep_kernel(Dims d, int B, const T* __restrict__ feats, const int32_t* __restrict__ n_acc,
                   const int64_t* __restrict__ pos, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ row_req, int64_t* __restrict__ row_pos,
                   int32_t* __restrict__ tags, T* __restrict__ packed, int32_t* __restrict__ err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = blockIdx.y;
  const int lim = d.S + 1;
  __shared__ int s_off, s_n;
  if (threadIdx.x < 32) {
    // offset of request b = sum of the valid counts before it (warp-parallel)
    int part = 0;
    for (int i = threadIdx.x; i < b; i += 32) {
      const int n = n_acc[i];
      part += (n >= 0 && n <= lim) ? n : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (threadIdx.x == 0) {
      const int n = n_acc[b];
      const bool ok = n >= 0 && n <= lim;
      if (!ok && t == 0) atomicOr(err, ERR_BAD_ACCEPTED);
      s_off = part;
      s_n = ok ? n : 0;
      if (t == 0) {
        offsets[b] = part;
        if (b == B - 1) offsets[B] = part + s_n;
      }
    }
  }
  __syncthreads();
  if (t >= s_n) return;
  const int r = s_off + t;
  const long long p = __ldcg(&pos[b]) + t;
  if (threadIdx.x == 0) {
    row_req[r] = b;
    row_pos[r] = p;
    tags[(size_t)b * d.W + (int)(p % d.W)] = (int32_t)p;
  }
  // gather the row: 16-byte chunks, loads batched ahead of the stores
  const uint4* src = reinterpret_cast<const uint4*>(feats + ((size_t)b * lim + t) * d.D);
  uint4* dst = reinterpret_cast<uint4*>(packed + (size_t)r * d.D);
  const int nchunk = d.D * (int)sizeof(T) / 16;
  for (int i0 = threadIdx.x; i0 < nchunk; i0 += 4 * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < nchunk) v[u] = __ldg(&src[i]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < nchunk) dst[i] = v[u];
    }
  }
}

// grid (Hm * qsplit, B, L): CTA (h, q) takes 1/qsplit of the state of one
// (layer, request, head), reads it once (all loads in flight together),
// advances it over the request's accepted rows in order, and writes it once.
__global__ void __launch_bounds__(256)
commit_state_kernel(Dims d, int qsplit, const int32_t* __restrict__ offsets,
                    const float* __restrict__ xbd, long long xls,
                    const float* __restrict__ A_log, float* __restrict__ state,
                    int64_t* __restrict__ pos) {
  extern __shared__ __align__(16) float sm[];
  pdl_trigger();
  pdl_wait();
  const int hd = blockIdx.x / qsplit, qs = blockIdx.x % qsplit;
  const int b = blockIdx.y, l = blockIdx.z;
  const int off = __ldcg(&offsets[b]), n = __ldcg(&offsets[b + 1]) - off;
  if (n <= 0) return;
  if (l == 0 && hd == 0 && qs == 0 && threadIdx.x == 0) pos[b] += n;
  const int P = d.P, N = d.N;
  float4* h = reinterpret_cast<float4*>(state + ((((size_t)l * d.Bmax + b) * d.Hm + hd) * P) * N);
  const int nq = P * N / 4;
  const int q0 = qs * (QPT * (int)blockDim.x);
  float4 hv[QPT];
  int pi[QPT], ci[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int q = q0 + threadIdx.x + u * blockDim.x;
    hv[u] = q < nq ? __ldcg(&h[q]) : make_float4(0.f, 0.f, 0.f, 0.f);
    pi[u] = (q * 4) / N;
    ci[u] = (q * 4) % N;
  }
  // stage x (this head), B and dt of the n accepted rows
  const int rows = d.S + 1;       // n <= block + 1
  float* sx = sm;                 // [rows][P]
  float* sb = sx + rows * P;      // [rows][N]
  float* sd = sb + rows * N;      // [rows]
  const float* xb = xbd + (size_t)l * xls;
  for (int i = threadIdx.x; i < n * (P / 4); i += blockDim.x) {
    const int t = i / (P / 4), c = (i % (P / 4)) * 4;
    *reinterpret_cast<float4*>(&sx[t * P + c]) =
        __ldcg(reinterpret_cast<const float4*>(xb + (size_t)(off + t) * d.NS + hd * P + c));
  }
  for (int i = threadIdx.x; i < n * (N / 4); i += blockDim.x) {
    const int t = i / (N / 4), c = (i % (N / 4)) * 4;
    *reinterpret_cast<float4*>(&sb[t * N + c]) =
        __ldcg(reinterpret_cast<const float4*>(xb + (size_t)(off + t) * d.NS + d.dinner + c));
  }
  for (int t = threadIdx.x; t < n; t += blockDim.x)
    sd[t] = __ldcg(&xb[(size_t)(off + t) * d.NS + d.dinner + N + hd]);
  __syncthreads();
  const float A = -expf(__ldcg(&A_log[l * d.Hm + hd]));
  for (int t = 0; t < n; ++t) {
    const float dt = sd[t];
    const float dec = expf(dt * A);
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const float xv = dt * sx[t * P + pi[u]];
      const float4 Bv = *reinterpret_cast<const float4*>(&sb[t * N + ci[u]]);
      hv[u].x = fmaf(dec, hv[u].x, xv * Bv.x);
      hv[u].y = fmaf(dec, hv[u].y, xv * Bv.y);
      hv[u].z = fmaf(dec, hv[u].z, xv * Bv.z);
      hv[u].w = fmaf(dec, hv[u].w, xv * Bv.w);
    }
  }
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int q = q0 + threadIdx.x + u * blockDim.x;
    if (q < nq) h[q] = hv[u];
  }
}

}  // namespace

cudaError_t launch_commit_prep(int dtype, const Dims& d, int B, const void* feats,
                               const int32_t* n_acc, const int64_t* pos, int32_t* offsets,
                               int32_t* row_req, int64_t* row_pos, int32_t* tags, void* packed,
                               int32_t* err, cudaStream_t st) {
  const dim3 grid(B, d.S + 1);
  if (dtype == HF_F32)
    return launch_pdl(commit_prep_kernel<float>, grid, dim3(128), 0, st, d, B,
                      (const float*)feats, n_acc, pos, offsets, row_req, row_pos, tags,
                      (float*)packed, err);
  return launch_pdl(commit_prep_kernel<__nv_bfloat16>, grid, dim3(128), 0, st, d, B,
                    (const __nv_bfloat16*)feats, n_acc, pos, offsets, row_req, row_pos, tags,
                    (__nv_bfloat16*)packed, err);
}

cudaError_t launch_commit_state(const Dims& d, int B, const int32_t* offsets, const float* xbd,
                                long long xls, const float* A_log, float* state, int64_t* pos,
                                cudaStream_t st) {
  // staging for block+1 rows of x (P values), B (N values) and dt
  const size_t smem = (size_t)(d.S + 1) * (d.P + d.N + 1) * sizeof(float);
  const int nq = d.P * d.N / 4;
  const int qsplit = (nq + QPT * 256 - 1) / (QPT * 256);
  return launch_pdl(commit_state_kernel, dim3(d.Hm * qsplit, B, d.L), dim3(256), smem, st, d,
                    qsplit, offsets, xbd, xls, A_log, state, pos);
}

}  // namespace hf
