// Window + block attention, split over the window with the splits combined
// through global memory: the variant behind hf_attention_noalloc.
//
// Attention (learnaivisually explainer, "That is HyFlash"): the 7 slot
// queries of a request attend, bidirectionally and with no mask, over the
// valid entries of that request's window ring and over the 7 slot keys.
// CTA (request b, KV head g, split j) takes ring slots [32 j, 32 j + 32) of
// (b, g) and all G = Hq/Hkv query heads sharing g (G*7 query rows): one bulk
// copy (TMA) per K/V tile into shared memory, converted to padded fp32 rows;
// scores, an exp2-based softmax and the P.V product in fp32. Each split
// writes (max, sum, partial O) to scratch memory; the last split of (b, g)
// to finish -- a ticket counter, no waiting -- combines all splits in split
// order (deterministic) and writes O. The scratch and tickets live in fixed
// device arrays (see the end of this file). hf_draft uses the cluster
// variant in attention_cluster.cu, which keeps the partials on chip.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace hf {
namespace {

constexpr int JT = 32;       // ring keys per split
constexpr int MAXS = 16;     // max block slots
constexpr int THREADS = 256;

struct AttnArgs {
  Dims d;
  int B;          // requests
  int nsplit;     // ring splits per (request, KV head)
  int n_attn;     // CTAs: B * Hkv * nsplit
  float qscale;   // log2(e) / sqrt(dh)
  const float* proj;    // [B*S, Nd] fp32: Q | K_s | V_s | C_s
  const void* ring_k;   // [B][Hkv][W][dh] of this layer
  const void* ring_v;
  const int64_t* pos;   // [B]
  void* mix;            // [B*S, Nz]: O at columns [0, Hq*dh)
  float* part_o;        // [B*Hkv*nsplit][R][dh]
  float* part_ml;       // [B*Hkv*nsplit][R][2]
  int* tickets;         // [B*Hkv], left at zero
  int32_t* err;         // ERR_TIMEOUT is ORed in here on a wait that gave up
  long long wait;       // limit (clock cycles) of the ring-tile wait
};

struct AttnSmem {
  size_t bar, stage_k, stage_v, q, k, v, s, w, flag, total;
};

__host__ __device__ inline AttnSmem attn_smem(const Dims& d, int esize, int nsplit) {
  AttnSmem m{};
  size_t off = 0;
  const int R = d.G * d.S, dhp = d.dh + 4, JK = JT + d.S;
  m.bar = off;
  off += 16;
  const size_t tile = (size_t)JT * d.dh * esize;
  m.stage_k = off;
  off += tile;
  m.stage_v = off;
  off += tile;
  m.q = off;
  off += (size_t)R * dhp * 4;
  m.k = off;
  off += (size_t)JK * dhp * 4;
  m.v = off;
  off += (size_t)JK * dhp * 4;
  m.s = off;
  off += (size_t)R * JK * 4;
  m.w = off;
  off += (size_t)nsplit * R * 4;
  off = (off + 15) & ~(size_t)15;
  m.flag = off;
  off += 16;
  m.total = off;
  return m;
}

template <typename T>
__device__ __forceinline__ void attn_cta(const AttnArgs& a, uint8_t* sm, int idx) {
  const Dims& d = a.d;
  const int split = idx % a.nsplit, rest = idx / a.nsplit;
  const int kvh = rest % d.Hkv, b = rest / d.Hkv;
  const int S = d.S, G = d.G, R = G * S, dh = d.dh, dhp = dh + 4, JK = JT + S;
  const AttnSmem L = attn_smem(d, (int)sizeof(T), a.nsplit);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);
  T* stk = reinterpret_cast<T*>(sm + L.stage_k);
  T* stv = reinterpret_cast<T*>(sm + L.stage_v);
  float* q = reinterpret_cast<float*>(sm + L.q);
  float* k = reinterpret_cast<float*>(sm + L.k);
  float* v = reinterpret_cast<float*>(sm + L.v);
  float* s = reinterpret_cast<float*>(sm + L.s);
  float* w = reinterpret_cast<float*>(sm + L.w);
  int* flag = reinterpret_cast<int*>(sm + L.flag);
  const int tid = threadIdx.x, nthr = blockDim.x;

  pdl_wait();
  const long long p = __ldcg(&a.pos[b]);
  const int nv = (int)(p < (long long)d.W ? p : (long long)d.W);
  const int j0 = split * JT;
  int nring = max(0, min(nv, j0 + JT) - j0);
  const int nslot = split == 0 ? S : 0;
  const size_t rowbase = (size_t)b * S;
  const size_t rb = ((size_t)b * d.Hkv + kvh) * d.W * dh;

  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (nring > 0) {
      const uint32_t bytes = (uint32_t)(nring * dh * sizeof(T));
      mbar_expect_tx(bar, 2 * bytes);
      bulk_g2s(stk, static_cast<const T*>(a.ring_k) + rb + (size_t)j0 * dh, bytes, bar);
      bulk_g2s(stv, static_cast<const T*>(a.ring_v) + rb + (size_t)j0 * dh, bytes, bar);
    }
  }
  // Query rows (pre-scaled), 16-byte loads.
  const int c4n = dh / 4;
  for (int i = tid; i < R * c4n; i += nthr) {
    const int r = i / c4n, c = (i % c4n) * 4, g = r / S, sl = r % S;
    float4 x = __ldcg(reinterpret_cast<const float4*>(
        a.proj + (rowbase + sl) * d.Nd + (size_t)(kvh * G + g) * dh + c));
    x.x *= a.qscale;
    x.y *= a.qscale;
    x.z *= a.qscale;
    x.w *= a.qscale;
    *reinterpret_cast<float4*>(&q[r * dhp + c]) = x;
  }
  __syncthreads();  // barrier initialised before anyone waits on it
  bool ok = true;
  if (nring > 0) ok = mbar_wait_for(bar, 0, a.wait);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) {
      if (a.err) atomicOr(a.err, ERR_TIMEOUT);
      // bounded, default limit: let the copies land before the stage buffers
      // are released (they are not read again on this path)
      mbar_wait(bar, 0);
    }
    nring = 0;  // the window tile is left out; the slot keys (split 0) stay
  } else if (nring > 0) {
    constexpr int VE = 16 / (int)sizeof(T);
    for (int i = tid; i < nring * dh / VE; i += nthr) {
      const int e0 = i * VE, j = e0 / dh, c = e0 % dh;
      const uint4 rk = *reinterpret_cast<const uint4*>(&stk[e0]);
      const uint4 rv = *reinterpret_cast<const uint4*>(&stv[e0]);
      const T* tk = reinterpret_cast<const T*>(&rk);
      const T* tv = reinterpret_cast<const T*>(&rv);
#pragma unroll
      for (int u = 0; u < VE; ++u) {
        k[j * dhp + c + u] = to_f(tk[u]);
        v[j * dhp + c + u] = to_f(tv[u]);
      }
    }
  }
  // slot keys/values after the ring rows (split 0 only)
  for (int i = tid; i < nslot * c4n; i += nthr) {
    const int j = i / c4n, c = (i % c4n) * 4;
    const float* row = a.proj + (rowbase + j) * d.Nd;
    *reinterpret_cast<float4*>(&k[(nring + j) * dhp + c]) =
        __ldcg(reinterpret_cast<const float4*>(row + d.QD + kvh * dh + c));
    *reinterpret_cast<float4*>(&v[(nring + j) * dhp + c]) =
        __ldcg(reinterpret_cast<const float4*>(row + d.QD + d.KVD + kvh * dh + c));
  }
  const int nk = nring + nslot;
  __syncthreads();

  for (int i = tid; i < R * nk; i += nthr) {
    const int r = i / nk, j = i % nk;
    float acc = 0.f;
    for (int dd = 0; dd < dh; dd += 4) {
      const float4 x = *reinterpret_cast<const float4*>(&q[r * dhp + dd]);
      const float4 y = *reinterpret_cast<const float4*>(&k[j * dhp + dd]);
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
    }
    s[r * JK + j] = acc;
  }
  __syncthreads();

  const int warp = tid / 32, lane = tid % 32, nw = nthr / 32;
  const size_t pbase = ((size_t)(b * d.Hkv + kvh) * a.nsplit + split) * R;
  for (int r = warp; r < R; r += nw) {
    float m = -INFINITY;
    for (int j = lane; j < nk; j += 32) m = fmaxf(m, s[r * JK + j]);
    m = warp_max(m);
    float l = 0.f;
    for (int j = lane; j < nk; j += 32) {
      const float e = exp2f(s[r * JK + j] - m);
      s[r * JK + j] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      a.part_ml[(pbase + r) * 2 + 0] = m;
      a.part_ml[(pbase + r) * 2 + 1] = l;
    }
  }
  __syncthreads();

  for (int i = tid; i < R * c4n; i += nthr) {
    const int r = i / c4n, c = (i % c4n) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < nk; ++j) {
      const float pj = s[r * JK + j];
      const float4 y = *reinterpret_cast<const float4*>(&v[j * dhp + c]);
      acc.x = fmaf(pj, y.x, acc.x);
      acc.y = fmaf(pj, y.y, acc.y);
      acc.z = fmaf(pj, y.z, acc.z);
      acc.w = fmaf(pj, y.w, acc.w);
    }
    *reinterpret_cast<float4*>(&a.part_o[(pbase + r) * dh + c]) = acc;
  }

  // Ticket: the last split of (b, g) to finish combines.
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = atomicAdd(&a.tickets[b * d.Hkv + kvh], 1) == a.nsplit - 1;
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  const size_t base = (size_t)(b * d.Hkv + kvh) * a.nsplit * R;
  for (int r = tid; r < R; r += nthr) {
    float M = -INFINITY;
    for (int sp = 0; sp < a.nsplit; ++sp)
      M = fmaxf(M, __ldcg(&a.part_ml[(base + (size_t)sp * R + r) * 2]));
    float Lsum = 0.f;
    for (int sp = 0; sp < a.nsplit; ++sp) {
      const size_t e = base + (size_t)sp * R + r;
      const float ls = __ldcg(&a.part_ml[e * 2 + 1]);
      const float wt = ls > 0.f ? exp2f(__ldcg(&a.part_ml[e * 2]) - M) : 0.f;
      w[sp * R + r] = wt;
      Lsum = fmaf(ls, wt, Lsum);
    }
    const float inv = 1.f / Lsum;
    for (int sp = 0; sp < a.nsplit; ++sp) w[sp * R + r] *= inv;
  }
  __syncthreads();
  T* mix = static_cast<T*>(a.mix);
  for (int i = tid; i < R * c4n; i += nthr) {
    const int r = i / c4n, c = (i % c4n) * 4, g = r / S, sl = r % S;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int sp = 0; sp < a.nsplit; ++sp) {
      const float wt = w[sp * R + r];
      const float4 o = __ldcg(reinterpret_cast<const float4*>(
          &a.part_o[(base + (size_t)sp * R + r) * dh + c]));
      acc.x = fmaf(wt, o.x, acc.x);
      acc.y = fmaf(wt, o.y, acc.y);
      acc.z = fmaf(wt, o.z, acc.z);
      acc.w = fmaf(wt, o.w, acc.w);
    }
    T* dst = mix + ((size_t)b * S + sl) * d.Nz + (size_t)(kvh * G + g) * dh + c;
    dst[0] = from_f<T>(acc.x);
    dst[1] = from_f<T>(acc.y);
    dst[2] = from_f<T>(acc.z);
    dst[3] = from_f<T>(acc.w);
  }
  if (tid == 0) a.tickets[b * d.Hkv + kvh] = 0;
}

template <typename T>
__global__ void __launch_bounds__(THREADS) attn_mem_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  pdl_trigger();
  attn_cta<T>(a, sm, blockIdx.x);
}

constexpr int kMaxDevices = 64;
// Dynamic shared memory the kernels were opened up to, per device (the
// attribute is a per-device setting of the function).
int g_configured_smem[kMaxDevices] = {};
std::mutex g_config_mu;

cudaError_t ensure_smem(int dev, size_t smem) {
  std::lock_guard<std::mutex> lock(g_config_mu);
  if ((int)smem <= g_configured_smem[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_mem_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_mem_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) g_configured_smem[dev] = (int)smem;
  return e;
}

cudaError_t launch(int dtype, const AttnArgs& a, cudaStream_t st) {
  const AttnSmem L = attn_smem(a.d, dtype == HF_F32 ? 4 : 2, a.nsplit);
  const dim3 grid(a.n_attn);
  if (dtype == HF_F32) return launch_pdl(attn_mem_kernel<float>, grid, dim3(THREADS), L.total, st, a);
  return launch_pdl(attn_mem_kernel<__nv_bfloat16>, grid, dim3(THREADS), L.total, st, a);
}

}  // namespace

// ---------------------------------------------------------------------------
// Allocation-free variant of the window+block attention.
//
// Some callers cannot allocate device memory at the moment they need this
// op: code running under an arena that owns all of the GPU's memory, a
// serving loop whose memory was sized once at start-up, or a host that must
// not trigger the device-wide synchronisation cudaMalloc/cudaFree can cause.
// For them the split partials and split tickets live in fixed arrays in the
// library's own device image instead of in a handle's scratch. The arrays
// exist on every GPU that loads the library, from load until the process
// exits. Tickets start at zero (static storage) and every call leaves them
// at zero.
namespace {

constexpr size_t kNoAllocFloats = (size_t)4 << 20;  // 16 MiB of fp32 partials
constexpr int kNoAllocTickets = 1 << 14;            // (request, KV head) pairs
static __device__ __align__(256) float g_noalloc_attn_scratch[kNoAllocFloats];
static __device__ __align__(256) int g_noalloc_attn_tickets[kNoAllocTickets];

struct NoAllocPtrs {
  float* scratch;
  int* tickets;
  int smem_optin;  // the device's opt-in shared memory per block
};
NoAllocPtrs g_noalloc[kMaxDevices] = {};
std::mutex g_noalloc_mu;
// limit of the ring-tile waits (hf_debug_set_wait_limit with no handle)
std::atomic<long long> g_noalloc_wait{kWaitCycles};

// The arrays' device addresses on the current device, looked up once per
// device (host code must not use the arrays' names as device pointers).
cudaError_t noalloc_scratch(int* dev_out, NoAllocPtrs* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc[dev].scratch) {
    void *p = nullptr, *t = nullptr;
    int optin = 0;
    e = cudaGetSymbolAddress(&p, g_noalloc_attn_scratch);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&t, g_noalloc_attn_tickets);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    g_noalloc[dev] = {static_cast<float*>(p), static_cast<int*>(t), optin};
  }
  *dev_out = dev;
  *out = g_noalloc[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace hf

extern "C" hf_status hf_attention_noalloc(int32_t dtype, int32_t batch, int32_t n_q_heads,
                                          int32_t n_kv_heads, int32_t head_dim, int32_t window,
                                          int32_t block, const float* proj, int32_t proj_ld,
                                          const void* ring_k, const void* ring_v,
                                          const int64_t* pos, void* out, int32_t out_ld,
                                          int32_t* status, void* stream) {
  using namespace hf;
  auto bad = [](const char* m) {
    set_thread_error(m);
    return HF_EINVAL;
  };
  if (dtype != HF_F32 && dtype != HF_BF16) return bad("dtype must be HF_F32 or HF_BF16");
  if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || window <= 0 || block <= 0)
    return bad("dimensions must be positive (batch >= 0)");
  if (n_q_heads % n_kv_heads) return bad("n_kv_heads must divide n_q_heads");
  if (head_dim % 8 || head_dim > 256) return bad("head_dim must be a multiple of 8, <= 256");
  if (block > MAXS || (n_q_heads / n_kv_heads) * block > 64)
    return bad("block must be <= 16 and (n_q_heads/n_kv_heads)*block <= 64");
  const long long qd = (long long)n_q_heads * head_dim, kvd = (long long)n_kv_heads * head_dim;
  if (proj_ld < qd + 2 * kvd || proj_ld % 4)
    return bad("proj_ld must be a multiple of 4 and >= Hq*dh + 2*Hkv*dh");
  if (out_ld < qd) return bad("out_ld must be >= Hq*dh");
  if (batch == 0) return HF_OK;
  if (!proj || !ring_k || !ring_v || !pos || !out) return bad("NULL buffer");
  if (reinterpret_cast<uintptr_t>(proj) % 16 || reinterpret_cast<uintptr_t>(ring_k) % 16 ||
      reinterpret_cast<uintptr_t>(ring_v) % 16)
    return bad("proj, ring_k and ring_v must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(status) % 4) return bad("status must be 4-byte aligned");
  const int nsplit = (window + JT - 1) / JT;
  const long long R = (long long)(n_q_heads / n_kv_heads) * block;
  const long long need = (long long)batch * n_kv_heads * nsplit * R * (head_dim + 2);
  if (need > (long long)kNoAllocFloats || (long long)batch * n_kv_heads > kNoAllocTickets) {
    char m[240];
    snprintf(m, sizeof m,
             "hf_attention_noalloc: needs %lld floats of scratch, the fixed array holds %zu "
             "(batch * n_kv_heads * ceil(window/32) * (Hq/Hkv) * block * (head_dim + 2)); "
             "batch * n_kv_heads must be <= %d",
             need, kNoAllocFloats, kNoAllocTickets);
    set_thread_error(m);
    return HF_EINVAL;
  }
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
  d.Hm = 1;
  d.P = 4;
  d.N = 4;
  d.esize = dtype == HF_F32 ? 4 : 2;
  const AttnSmem L = attn_smem(d, d.esize, nsplit);
  int dev = 0;
  NoAllocPtrs ptrs{};
  cudaError_t e = noalloc_scratch(&dev, &ptrs);
  if (e == cudaSuccess && L.total > (size_t)ptrs.smem_optin) {
    char m[240];
    snprintf(m, sizeof m,
             "hf_attention_noalloc: a CTA needs %zu bytes of shared memory, the device allows %d "
             "(it grows with (Hq/Hkv)*block*head_dim and with window/32)",
             L.total, ptrs.smem_optin);
    set_thread_error(m);
    return HF_EINVAL;
  }
  if (e == cudaSuccess) e = ensure_smem(dev, L.total);
  if (e == cudaSuccess) {
    AttnArgs a{};
    a.d = d;
    a.B = batch;
    a.nsplit = nsplit;
    a.n_attn = batch * n_kv_heads * nsplit;
    a.qscale = 1.4426950408889634f / sqrtf((float)head_dim);
    a.proj = proj;
    a.ring_k = ring_k;
    a.ring_v = ring_v;
    a.pos = pos;
    a.mix = out;
    a.part_o = ptrs.scratch;
    a.part_ml = ptrs.scratch + (size_t)a.n_attn * R * head_dim;
    a.tickets = ptrs.tickets;
    a.err = status;
    a.wait = g_noalloc_wait.load();
    e = launch(dtype, a, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) {
    set_thread_error(cudaGetErrorString(e));
    return HF_ECUDA;
  }
  return HF_OK;
}

namespace hf {
void set_noalloc_wait_limit(long long cycles) { g_noalloc_wait.store(cycles); }
}  // namespace hf
