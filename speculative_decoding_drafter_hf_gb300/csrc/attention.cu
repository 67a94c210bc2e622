// Window + block attention and the draft-time memory read for one layer.
//
// Attention (learnaivisually explainer, "That is HyFlash"): the 7 slot
// queries of a request attend, bidirectionally and with no mask, over the
// valid entries of that request's window ring and over the 7 slot keys. One
// CTA takes one (request, KV head, window split) and all G = Hq/Hkv query
// heads that share the KV head (G*7 query rows), so each K/V tile is read
// from HBM once. Splits combine with the usual max/sum rescaling, in a fixed
// order, in a second kernel.
//
// Memory read: y[s, h, p] = sum_n state[h, p, n] * C_s[s, n], with C_s the
// slot projection through W_C; the state is only read.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace hf {
namespace {

constexpr int JT = 32;      // ring keys per split
constexpr int MAXS = 16;    // max block slots

template <typename T>
__global__ void __launch_bounds__(128)
attn_partial_kernel(Dims d, const float* __restrict__ proj, const T* __restrict__ ring_k,
                    const T* __restrict__ ring_v, const int64_t* __restrict__ pos,
                    float* __restrict__ part_o, float* __restrict__ part_ml, int nsplit,
                    float qscale) {
  extern __shared__ __align__(16) float sm[];
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int S = d.S, G = d.G, R = G * S, dh = d.dh, dhp = dh + 4, JK = JT + S;
  float* q = sm;
  float* k = q + R * dhp;
  float* v = k + JK * dhp;
  float* s = v + JK * dhp;
  const int tid = threadIdx.x, nthr = blockDim.x;

  const long long p = pos[b];
  const int nv = (int)(p < (long long)d.W ? p : (long long)d.W);
  const int j0 = split * JT;
  const int nring = max(0, min(nv, j0 + JT) - j0);
  const int nslot = split == 0 ? S : 0;
  const int nk = nring + nslot;
  const size_t rowbase = (size_t)b * S;

  for (int i = tid; i < R * dh; i += nthr) {
    int r = i / dh, dd = i % dh, g = r / S, sl = r % S;
    q[r * dhp + dd] = proj[(rowbase + sl) * d.Nd + (size_t)(kvh * G + g) * dh + dd] * qscale;
  }
  const size_t rb = ((size_t)b * d.Hkv + kvh) * d.W * dh;
  for (int i = tid; i < nring * dh; i += nthr) {
    int j = i / dh, dd = i % dh;
    k[j * dhp + dd] = to_f(ring_k[rb + (size_t)(j0 + j) * dh + dd]);
    v[j * dhp + dd] = to_f(ring_v[rb + (size_t)(j0 + j) * dh + dd]);
  }
  for (int i = tid; i < nslot * dh; i += nthr) {
    int j = i / dh, dd = i % dh;
    const float* row = proj + (rowbase + j) * d.Nd;
    k[(nring + j) * dhp + dd] = row[d.QD + kvh * dh + dd];
    v[(nring + j) * dhp + dd] = row[d.QD + d.KVD + kvh * dh + dd];
  }
  __syncthreads();

  for (int i = tid; i < R * nk; i += nthr) {
    int r = i / nk, j = i % nk;
    float acc = 0.f;
    for (int dd = 0; dd < dh; dd += 4) {
      float4 a = *reinterpret_cast<const float4*>(&q[r * dhp + dd]);
      float4 c = *reinterpret_cast<const float4*>(&k[j * dhp + dd]);
      acc = fmaf(a.x, c.x, fmaf(a.y, c.y, fmaf(a.z, c.z, fmaf(a.w, c.w, acc))));
    }
    s[r * JK + j] = acc;
  }
  __syncthreads();

  const int warp = tid / 32, lane = tid % 32, nw = nthr / 32;
  const size_t pbase = ((size_t)(b * d.Hkv + kvh) * nsplit + split) * R;
  for (int r = warp; r < R; r += nw) {
    float m = -INFINITY;
    for (int j = lane; j < nk; j += 32) m = fmaxf(m, s[r * JK + j]);
    m = warp_max(m);
    float l = 0.f;
    for (int j = lane; j < nk; j += 32) {
      float e = exp2f(s[r * JK + j] - m);
      s[r * JK + j] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      part_ml[(pbase + r) * 2 + 0] = m;
      part_ml[(pbase + r) * 2 + 1] = l;
    }
  }
  __syncthreads();

  const int d4n = dh / 4;
  for (int i = tid; i < R * d4n; i += nthr) {
    int r = i / d4n, d4 = (i % d4n) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < nk; ++j) {
      float pj = s[r * JK + j];
      float4 vv = *reinterpret_cast<const float4*>(&v[j * dhp + d4]);
      acc.x = fmaf(pj, vv.x, acc.x);
      acc.y = fmaf(pj, vv.y, acc.y);
      acc.z = fmaf(pj, vv.z, acc.z);
      acc.w = fmaf(pj, vv.w, acc.w);
    }
    *reinterpret_cast<float4*>(&part_o[(pbase + r) * dh + d4]) = acc;
  }
}

template <typename T>
__global__ void attn_combine_kernel(Dims d, const float* __restrict__ part_o,
                                    const float* __restrict__ part_ml, int nsplit,
                                    T* __restrict__ mix) {
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int S = d.S, G = d.G, R = G * S, dh = d.dh;
  const size_t base = (size_t)(b * d.Hkv + kvh) * nsplit * R;
  for (int i = threadIdx.x; i < R * dh; i += blockDim.x) {
    int r = i / dh, dd = i % dh;
    float M = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, part_ml[(base + (size_t)sp * R + r) * 2]);
    float L = 0.f, acc = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
      size_t e = base + (size_t)sp * R + r;
      float ls = part_ml[e * 2 + 1];
      if (ls > 0.f) {
        float w = exp2f(part_ml[e * 2] - M);
        L = fmaf(ls, w, L);
        acc = fmaf(part_o[e * dh + dd], w, acc);
      }
    }
    int g = r / S, sl = r % S;
    mix[((size_t)b * S + sl) * d.Nz + (size_t)(kvh * G + g) * dh + dd] = from_f<T>(acc / L);
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
memread_kernel(Dims d, const float* __restrict__ proj, const float* __restrict__ state,
               T* __restrict__ mix) {
  __shared__ float cs[MAXS * 256];
  const int hd = blockIdx.x, b = blockIdx.y;
  const int S = d.S, N = d.N, P = d.P;
  const int cC = d.QD + 2 * d.KVD;
  for (int i = threadIdx.x; i < S * N; i += blockDim.x) {
    int sl = i / N, n = i % N;
    cs[sl * N + n] = proj[((size_t)b * S + sl) * d.Nd + cC + n];
  }
  __syncthreads();
  const float* h = state + (((size_t)b * d.Hm + hd) * P) * N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  for (int p = warp; p < P; p += nw) {
    float acc[MAXS];
#pragma unroll
    for (int sl = 0; sl < MAXS; ++sl) acc[sl] = 0.f;
    for (int n = lane; n < N; n += 32) {
      float hv = h[(size_t)p * N + n];
#pragma unroll
      for (int sl = 0; sl < MAXS; ++sl)
        if (sl < S) acc[sl] = fmaf(hv, cs[sl * N + n], acc[sl]);
    }
#pragma unroll
    for (int sl = 0; sl < MAXS; ++sl) {
      if (sl < S) {
        float v = warp_sum(acc[sl]);
        if (lane == 0)
          mix[((size_t)b * S + sl) * d.Nz + d.QD + (size_t)hd * P + p] = from_f<T>(v);
      }
    }
  }
}

template <typename T>
cudaError_t run(const Dims& d, int B, const float* proj, const void* ring_k, const void* ring_v,
                const int64_t* pos, const float* state, void* mix, float* part_o,
                float* part_ml, int nsplit, cudaStream_t st, int* la, int* lo) {
  if (B <= 0) return cudaSuccess;
  const int R = d.G * d.S, dhp = d.dh + 4, JK = JT + d.S;
  size_t smem = (size_t)(R * dhp + 2 * JK * dhp + R * JK) * sizeof(float);
  const float qscale = 1.4426950408889634f / sqrtf((float)d.dh);
  attn_partial_kernel<T><<<dim3(nsplit, d.Hkv, B), 128, smem, st>>>(
      d, proj, (const T*)ring_k, (const T*)ring_v, pos, part_o, part_ml, nsplit, qscale);
  ++*la;
  memread_kernel<T><<<dim3(d.Hm, B), 256, 0, st>>>(d, proj, state, (T*)mix);
  ++*la;
  attn_combine_kernel<T><<<dim3(d.Hkv, B), 256, 0, st>>>(d, part_o, part_ml, nsplit, (T*)mix);
  ++*lo;
  return cudaGetLastError();
}

}  // namespace

// Dynamic shared memory of the attention kernel is raised once per process
// (at handle creation), so launches stay legal inside stream capture.
cudaError_t configure_attn(const Dims& d) {
  const int R = d.G * d.S, dhp = d.dh + 4, JK = JT + d.S;
  const int smem = (int)((size_t)(R * dhp + 2 * JK * dhp + R * JK) * sizeof(float));
  static int configured = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (smem <= configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_partial_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) configured = smem;
  return e;
}

cudaError_t launch_attn_mem(int dtype, const Dims& d, int B, const float* proj,
                            const void* ring_k, const void* ring_v, const int64_t* pos,
                            const float* state, void* mix, float* part_o, float* part_ml,
                            int nsplit, cudaStream_t st, int* la, int* lo) {
  if (dtype == HF_F32)
    return run<float>(d, B, proj, ring_k, ring_v, pos, state, mix, part_o, part_ml, nsplit, st,
                      la, lo);
  return run<__nv_bfloat16>(d, B, proj, ring_k, ring_v, pos, state, mix, part_o, part_ml, nsplit,
                            st, la, lo);
}

}  // namespace hf

// ---------------------------------------------------------------------------
// Allocation-free variant of the window+block attention.
//
// Some callers cannot allocate device memory at the moment they need this
// op: code running under an arena that owns all of the GPU's memory, a
// serving loop whose memory was sized once at start-up, or a host that must
// not trigger the device-wide synchronisation cudaMalloc/cudaFree can cause.
// For them the split partials live in one fixed array in the library's own
// device image instead of in a handle's scratch. The array exists on every
// GPU that loads the library, from load until the process exits.
namespace hf {
namespace {

constexpr size_t kNoAllocFloats = (size_t)4 << 20;  // 16 MiB of fp32 partials
static __device__ __align__(256) float g_noalloc_attn_scratch[kNoAllocFloats];

constexpr int kMaxDevices = 64;
float* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// The symbol's device address on the current device, looked up once per
// device (host code must not use the array's name as a device pointer).
cudaError_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_attn_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

template <typename T>
cudaError_t run_noalloc(const Dims& d, int B, const float* proj, const void* ring_k,
                        const void* ring_v, const int64_t* pos, void* out, int nsplit,
                        float* scratch, cudaStream_t st) {
  const int R = d.G * d.S, dhp = d.dh + 4, JK = JT + d.S;
  const size_t n_o = (size_t)B * d.Hkv * nsplit * R * d.dh;
  float* part_o = scratch;
  float* part_ml = scratch + n_o;
  size_t smem = (size_t)(R * dhp + 2 * JK * dhp + R * JK) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float qscale = 1.4426950408889634f / sqrtf((float)d.dh);
  attn_partial_kernel<T><<<dim3(nsplit, d.Hkv, B), 128, smem, st>>>(
      d, proj, (const T*)ring_k, (const T*)ring_v, pos, part_o, part_ml, nsplit, qscale);
  attn_combine_kernel<T><<<dim3(d.Hkv, B), 256, 0, st>>>(d, part_o, part_ml, nsplit, (T*)out);
  return cudaGetLastError();
}

}  // namespace
}  // namespace hf

extern "C" hf_status hf_attention_noalloc(int32_t dtype, int32_t batch, int32_t n_q_heads,
                                          int32_t n_kv_heads, int32_t head_dim, int32_t window,
                                          int32_t block, const float* proj, int32_t proj_ld,
                                          const void* ring_k, const void* ring_v,
                                          const int64_t* pos, void* out, int32_t out_ld,
                                          void* stream) {
  using namespace hf;
  auto bad = [](const char* m) {
    set_thread_error(m);
    return HF_EINVAL;
  };
  if (dtype != HF_F32 && dtype != HF_BF16) return bad("dtype must be HF_F32 or HF_BF16");
  if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || window <= 0 || block <= 0)
    return bad("dimensions must be positive (batch >= 0)");
  if (n_q_heads % n_kv_heads) return bad("n_kv_heads must divide n_q_heads");
  if (head_dim % 4 || head_dim > 256) return bad("head_dim must be a multiple of 4, <= 256");
  if (block > MAXS || (n_q_heads / n_kv_heads) * block > 64)
    return bad("block must be <= 16 and (n_q_heads/n_kv_heads)*block <= 64");
  const long long qd = (long long)n_q_heads * head_dim, kvd = (long long)n_kv_heads * head_dim;
  if (proj_ld < qd + 2 * kvd) return bad("proj_ld must be >= Hq*dh + 2*Hkv*dh");
  if (out_ld < qd) return bad("out_ld must be >= Hq*dh");
  if (batch == 0) return HF_OK;
  if (!proj || !ring_k || !ring_v || !pos || !out) return bad("NULL buffer");
  const int nsplit = (window + JT - 1) / JT;
  const long long R = (long long)(n_q_heads / n_kv_heads) * block;
  const long long need = (long long)batch * n_kv_heads * nsplit * R * (head_dim + 2);
  if (need > (long long)kNoAllocFloats) {
    char m[200];
    snprintf(m, sizeof m,
             "hf_attention_noalloc: needs %lld floats of scratch, the fixed array holds %zu "
             "(batch * n_kv_heads * ceil(window/32) * (Hq/Hkv) * block * (head_dim + 2))",
             need, kNoAllocFloats);
    set_thread_error(m);
    return HF_EINVAL;
  }
  float* scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e == cudaSuccess) {
    Dims d{};
    d.Hq = n_q_heads;
    d.Hkv = n_kv_heads;
    d.dh = head_dim;
    d.W = window;
    d.S = block;
    d.G = n_q_heads / n_kv_heads;
    d.QD = (int)qd;
    d.KVD = (int)kvd;
    d.Nd = proj_ld;
    d.Nz = out_ld;
    d.esize = dtype == HF_F32 ? 4 : 2;
    cudaStream_t st = (cudaStream_t)stream;
    e = dtype == HF_F32
            ? run_noalloc<float>(d, batch, proj, ring_k, ring_v, pos, out, nsplit, scratch, st)
            : run_noalloc<__nv_bfloat16>(d, batch, proj, ring_k, ring_v, pos, out, nsplit, scratch,
                                         st);
  }
  if (e != cudaSuccess) {
    set_thread_error(cudaGetErrorString(e));
    return HF_ECUDA;
  }
  return HF_OK;
}
