// Prefill helpers: reset a request, fill its window from the last W prefix
// features, the chunked decay scan of the memory fold, set its position.
// (The fold's contractions run on the tensor-core GEMM: gemm_tc.cu.)
//
// Source: HyFlash abstract ("recurrent memory compresses historical target
// features into fixed-size states") and the explainer's "That is HyFlash":
// the memory holds the compressed history of committed target features.
// Folding a prefix is committing all of its features at once, from h = 0.
#include "common.cuh"

namespace hf {
namespace {

// grid (blocks, n_req, L): zero the request's state (all layers), clear its
// ring tags and position.
__global__ void prefill_reset_kernel(Dims d, const int32_t* __restrict__ reqs,
                                     float* __restrict__ state, int32_t* __restrict__ tags,
                                     int64_t* __restrict__ pos) {
  const int b = reqs[blockIdx.y], l = blockIdx.z;
  const size_t per4 = (size_t)d.Hm * d.P * d.N / 4;
  float4* h = reinterpret_cast<float4*>(state + ((size_t)l * d.Bmax + b) * per4 * 4);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < per4;
       i += (size_t)gridDim.x * blockDim.x)
    h[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (blockIdx.x == 0 && l == 0) {
    for (int i = threadIdx.x; i < d.W; i += blockDim.x) tags[(size_t)b * d.W + i] = -1;
    if (threadIdx.x == 0) pos[b] = 0;
  }
}

// grid (n_rows): packed ring row j -> request i, its position, gathered row.
template <typename T>
__global__ void prefill_ring_prep_kernel(Dims d, int n_req, const int32_t* __restrict__ lens,
                                         const int32_t* __restrict__ reqs,
                                         const T* __restrict__ feats,
                                         int32_t* __restrict__ row_req,
                                         int64_t* __restrict__ row_pos,
                                         int32_t* __restrict__ tags, T* __restrict__ packed,
                                         int64_t* __restrict__ req_len) {
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
        if (req_len && jj == 0) req_len[b] = L;
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
  // D * sizeof(T) is a multiple of 16 and both rows are 16-byte aligned
  const uint4* src = reinterpret_cast<const uint4*>(feats + (size_t)s_src * d.D);
  uint4* dst = reinterpret_cast<uint4*>(packed + (size_t)j * d.D);
  for (int i = threadIdx.x; i < d.D * (int)sizeof(T) / 16; i += blockDim.x) dst[i] = src[i];
}

// grid (Hm), 32 warps: chunked suffix scan of a_t = dt_t * A_h over one
// segment. Warp w owns a contiguous range of whole chunks; pass 1 sums each
// range, a CTA-level suffix over the 32 range totals gives every warp the
// decay carried in from later tokens; pass 2 walks the warp's chunks from the
// last one back, with an inclusive suffix scan across lanes (shuffles) inside
// each chunk, and turns dt_t into w_t = dt_t * exp(sum_{s>t} a_s).
constexpr int DECAY_MAX_E = 8;  // tokens per lane per chunk (chunk <= 256)

__global__ void __launch_bounds__(1024)
prefill_decay_kernel(Dims d, int layer, int T, int ldt, int chunk, float* __restrict__ dtw,
                     const float* __restrict__ A_log, float* __restrict__ seg_decay) {
  __shared__ float wsum[32];
  const int h = blockIdx.x, warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float A = -expf(A_log[layer * d.Hm + h]);
  float* row = dtw + (size_t)h * ldt;
  const int per = (T + 31) / 32;
  const int R = (per + chunk - 1) / chunk * chunk;  // tokens per warp, whole chunks
  const int w0 = warp * R, w1 = min(T, w0 + R);
  float acc = 0.f;
  for (int t = w0 + lane; t < w1; t += 32) acc += row[t] * A;
  acc = warp_sum(acc);
  if (lane == 0) wsum[warp] = acc;
  __syncthreads();
  float carry = 0.f;  // sum over all tokens after this warp's range
  for (int w2 = 31; w2 > warp; --w2) carry += wsum[w2];
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w2 = 31; w2 >= 0; --w2) tot += wsum[w2];
    seg_decay[h] = expf(tot);
  }
  const int E = chunk / 32;
  for (int k = R / chunk - 1; k >= 0; --k) {
    const int cs = w0 + k * chunk;
    if (cs >= w1) continue;
    float a[DECAY_MAX_E], dv[DECAY_MAX_E];
    float lane_tot = 0.f;
#pragma unroll
    for (int e = 0; e < DECAY_MAX_E; ++e) {
      const int t = cs + lane * E + e;
      dv[e] = (e < E && t < w1) ? row[t] : 0.f;
      a[e] = dv[e] * A;
      lane_tot += a[e];
    }
    float incl = lane_tot;  // sum over this lane and all later lanes of the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += y;
    }
    float excl = __shfl_down_sync(0xffffffffu, incl, 1);  // later lanes only
    if (lane == 31) excl = 0.f;
    const float chunk_tot = __shfl_sync(0xffffffffu, incl, 0);
    float run = carry + excl;
#pragma unroll
    for (int e = DECAY_MAX_E - 1; e >= 0; --e) {
      const int t = cs + lane * E + e;
      if (e < E && t < w1) row[t] = dv[e] * expf(run);
      run += a[e];
    }
    carry += chunk_tot;
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
  const size_t per4 = (size_t)d.Hm * d.P * d.N / 4;
  const int blocks = (int)std::min<size_t>((per4 + 1023) / 1024, 64);
  prefill_reset_kernel<<<dim3(blocks, n_req, d.L), 256, 0, st>>>(d, reqs, state, tags, pos);
  return cudaGetLastError();
}

cudaError_t launch_prefill_ring_prep(int dtype, const Dims& d, int n_req, int n_rows,
                                     const int32_t* lens, const int32_t* reqs, const void* feats,
                                     int32_t* row_req, int64_t* row_pos, int32_t* tags,
                                     void* packed, int64_t* req_len, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (dtype == HF_F32)
    prefill_ring_prep_kernel<float><<<n_rows, 128, 0, st>>>(
        d, n_req, lens, reqs, (const float*)feats, row_req, row_pos, tags, (float*)packed,
        req_len);
  else
    prefill_ring_prep_kernel<__nv_bfloat16><<<n_rows, 128, 0, st>>>(
        d, n_req, lens, reqs, (const __nv_bfloat16*)feats, row_req, row_pos, tags,
        (__nv_bfloat16*)packed, req_len);
  return cudaGetLastError();
}

cudaError_t launch_prefill_decay(const Dims& d, int layer, int T, int ldt, int chunk, float* dtw,
                                 const float* A_log, float* seg_decay, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (chunk < 32 || chunk > 32 * DECAY_MAX_E || chunk % 32) return cudaErrorInvalidValue;
  prefill_decay_kernel<<<d.Hm, 1024, 0, st>>>(d, layer, T, ldt, chunk, dtw, A_log, seg_decay);
  return cudaGetLastError();
}

cudaError_t launch_prefill_finish(int n_req, const int32_t* lens, const int32_t* reqs,
                                  int64_t* pos, cudaStream_t st) {
  if (n_req <= 0) return cudaSuccess;
  prefill_finish_kernel<<<1, 256, 0, st>>>(n_req, lens, reqs, pos);
  return cudaGetLastError();
}

}  // namespace hf
