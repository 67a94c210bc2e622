// Commit path: the sequential memory update, with the accepted-count check,
// the packed offsets, the ring tags and the position update.
//
// Source: learnaivisually explainer, FAQ "Why does the memory update only
// from committed features?" and "That is HyFlash": after verification only
// the newly committed features update the state, in order; drafting never
// writes it. Ring slots follow the sliding-window rule (Jargon,
// "Sliding-window attention"): the window keeps the most recent W committed
// positions, position t in slot t mod W. The K/V ring append itself happens
// in the commit projection's epilogue (common.cuh, EPI_SSM_KV).
#include "common.cuh"

namespace hf {
namespace {

constexpr int QPT = 2;  // float4 state elements per thread of the state update

// grid (Hm * qsplit, B, L): CTA (h, q) takes 1/qsplit of the state of one
// (layer, request, head), reads it once (all loads in flight together),
// advances it over the request's accepted rows in order, and writes it once.
// CTA (0, b, 0) also checks n_b, writes offsets[b] (and offsets[B]), the ring
// tags of the appended positions, and pos[b] += n_b.
__global__ void __launch_bounds__(256)
commit_state_kernel(Dims d, int B, int qsplit, const int32_t* __restrict__ n_acc,
                    const float* __restrict__ xbd, long long xls,
                    const float* __restrict__ A_log, float* __restrict__ state,
                    int64_t* __restrict__ pos, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ tags, int32_t* __restrict__ err) {
  extern __shared__ __align__(16) float sm[];
  pdl_trigger();
  pdl_wait();
  const int hd = blockIdx.x / qsplit, qs = blockIdx.x % qsplit;
  const int b = blockIdx.y, l = blockIdx.z;
  const int lim = d.S + 1;
  const int n_raw = __ldcg(&n_acc[b]);
  const bool valid = n_raw >= 0 && n_raw <= lim;
  const int n = valid ? n_raw : 0;
  if (blockIdx.x == 0 && l == 0) {
    __shared__ long long s_pos;
    if (threadIdx.x < 32) {
      int part = 0;
      for (int i = threadIdx.x; i < b; i += 32) {
        const int m = __ldcg(&n_acc[i]);
        part += (m >= 0 && m <= lim) ? m : 0;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (threadIdx.x == 0) {
        if (!valid) atomicOr(err, ERR_BAD_ACCEPTED);
        offsets[b] = part;
        if (b == B - 1) offsets[B] = part + n;
        s_pos = __ldcg(&pos[b]);
      }
    }
    __syncthreads();
    const long long p0 = s_pos;
    for (int t = threadIdx.x; t < n; t += blockDim.x)
      tags[(size_t)b * d.W + (int)((p0 + t) % d.W)] = (int32_t)(p0 + t);
    if (threadIdx.x == 0) pos[b] = p0 + n;
  }
  if (n == 0) return;
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
  // stage x (this head), B and dt of the n accepted rows b*(S+1) + t
  float* sx = sm;             // [lim][P]
  float* sb = sx + lim * P;   // [lim][N]
  float* sd = sb + lim * N;   // [lim]
  const float* xb = xbd + (size_t)l * xls + (size_t)b * lim * d.NS;
  for (int i = threadIdx.x; i < n * (P / 4); i += blockDim.x) {
    const int t = i / (P / 4), c = (i % (P / 4)) * 4;
    *reinterpret_cast<float4*>(&sx[t * P + c]) =
        __ldcg(reinterpret_cast<const float4*>(xb + (size_t)t * d.NS + hd * P + c));
  }
  for (int i = threadIdx.x; i < n * (N / 4); i += blockDim.x) {
    const int t = i / (N / 4), c = (i % (N / 4)) * 4;
    *reinterpret_cast<float4*>(&sb[t * N + c]) =
        __ldcg(reinterpret_cast<const float4*>(xb + (size_t)t * d.NS + d.dinner + c));
  }
  for (int t = threadIdx.x; t < n; t += blockDim.x)
    sd[t] = __ldcg(&xb[(size_t)t * d.NS + d.dinner + N + hd]);
  __syncthreads();
  const float A = -expf(__ldg(&A_log[l * d.Hm + hd]));
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

cudaError_t launch_commit_state(const Dims& d, int B, const int32_t* n_acc, const float* xbd,
                                long long xls, const float* A_log, float* state, int64_t* pos,
                                int32_t* offsets, int32_t* tags, int32_t* err, cudaStream_t st) {
  // staging for block+1 rows of x (P values), B (N values) and dt
  const size_t smem = (size_t)(d.S + 1) * (d.P + d.N + 1) * sizeof(float);
  const int nq = d.P * d.N / 4;
  const int qsplit = (nq + QPT * 256 - 1) / (QPT * 256);
  return launch_pdl(commit_state_kernel, dim3(d.Hm * qsplit, B, d.L), dim3(256), smem, st, d, B,
                    qsplit, n_acc, xbd, xls, A_log, state, pos, offsets, tags, err);
}

}  // namespace hf
