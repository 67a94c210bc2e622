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

// grid (B, S+1): CTA (b, t) owns accepted row t of request b.
template <typename T>
__global__ void commit_prep_kernel(Dims d, int B, const T* __restrict__ feats,
                                   const int32_t* __restrict__ n_acc,
                                   const int64_t* __restrict__ pos, int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ row_req, int64_t* __restrict__ row_pos,
                                   int32_t* __restrict__ tags, T* __restrict__ packed,
                                   int32_t* __restrict__ err) {
  const int b = blockIdx.x, t = blockIdx.y;
  const int lim = d.S + 1;
  __shared__ int s_off, s_n;
  if (threadIdx.x == 0) {
    int off = 0;
    for (int i = 0; i < b; ++i) {
      int n = n_acc[i];
      off += (n >= 0 && n <= lim) ? n : 0;
    }
    int n = n_acc[b];
    bool ok = n >= 0 && n <= lim;
    if (!ok && t == 0) atomicOr(err, ERR_BAD_ACCEPTED);
    s_off = off;
    s_n = ok ? n : 0;
    if (t == 0) {
      offsets[b] = off;
      if (b == B - 1) offsets[B] = off + s_n;
    }
  }
  __syncthreads();
  if (t >= s_n) return;
  const int r = s_off + t;
  const long long p = pos[b] + t;
  if (threadIdx.x == 0) {
    row_req[r] = b;
    row_pos[r] = p;
    tags[(size_t)b * d.W + (int)(p % d.W)] = (int32_t)p;
  }
  const T* src = feats + ((size_t)b * lim + t) * d.D;
  T* dst = packed + (size_t)r * d.D;
  for (int i = threadIdx.x; i < d.D; i += blockDim.x) dst[i] = src[i];
}

// grid (Hm, B, L): the state of one (layer, request, head) is read once,
// advanced over the request's accepted rows in order, and written once.
__global__ void __launch_bounds__(256)
commit_state_kernel(Dims d, const int32_t* __restrict__ offsets, const float* __restrict__ xbd,
                    long long xls, const float* __restrict__ A_log, float* __restrict__ state,
                    int64_t* __restrict__ pos) {
  const int hd = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
  const int off = offsets[b], n = offsets[b + 1] - off;
  if (n <= 0) return;
  if (l == 0 && hd == 0 && threadIdx.x == 0) pos[b] += n;
  const float A = -expf(A_log[l * d.Hm + hd]);
  float4* h = reinterpret_cast<float4*>(state + ((((size_t)l * d.Bmax + b) * d.Hm + hd) * d.P) * d.N);
  const float* xb = xbd + (size_t)l * xls;
  const int nq = d.P * d.N / 4;
  for (int q = threadIdx.x; q < nq; q += blockDim.x) {
    const int e = q * 4, p = e / d.N, nn = e % d.N;
    float4 hv = h[q];
    for (int t = 0; t < n; ++t) {
      const float* row = xb + (size_t)(off + t) * d.NS;
      const float dt = row[d.dinner + d.N + hd];
      const float dec = expf(dt * A);
      const float xv = dt * row[hd * d.P + p];
      const float4 Bv = *reinterpret_cast<const float4*>(row + d.dinner + nn);
      hv.x = fmaf(dec, hv.x, xv * Bv.x);
      hv.y = fmaf(dec, hv.y, xv * Bv.y);
      hv.z = fmaf(dec, hv.z, xv * Bv.z);
      hv.w = fmaf(dec, hv.w, xv * Bv.w);
    }
    h[q] = hv;
  }
}

}  // namespace

cudaError_t launch_commit_prep(int dtype, const Dims& d, int B, const void* feats,
                               const int32_t* n_acc, const int64_t* pos, int32_t* offsets,
                               int32_t* row_req, int64_t* row_pos, int32_t* tags, void* packed,
                               int32_t* err, cudaStream_t st) {
  dim3 grid(B, d.S + 1);
  if (dtype == HF_F32)
    commit_prep_kernel<float><<<grid, 128, 0, st>>>(d, B, (const float*)feats, n_acc, pos,
                                                    offsets, row_req, row_pos, tags,
                                                    (float*)packed, err);
  else
    commit_prep_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(
        d, B, (const __nv_bfloat16*)feats, n_acc, pos, offsets, row_req, row_pos, tags,
        (__nv_bfloat16*)packed, err);
  return cudaGetLastError();
}

cudaError_t launch_commit_state(const Dims& d, int B, const int32_t* offsets, const float* xbd,
                                long long xls, const float* A_log, float* state, int64_t* pos,
                                cudaStream_t st) {
  commit_state_kernel<<<dim3(d.Hm, B, d.L), 256, 0, st>>>(d, offsets, xbd, xls, A_log, state,
                                                         pos);
  return cudaGetLastError();
}

}  // namespace hf
