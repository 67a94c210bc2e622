// Window + block attention and the draft-time memory read for one layer, in
// one launch; the path hf_draft takes.
//
// Attention (learnaivisually explainer, "That is HyFlash"): the 7 slot
// queries of a request attend, bidirectionally and with no mask, over the
// valid entries of that request's window ring and over the 7 slot keys.
//
// Work split: the window of (request b, KV head g) is cut into `nsplit` <= 8
// tiles of JT keys; the nsplit CTAs of (b, g) form one thread-block cluster.
// Each CTA takes all G = Hq/Hkv query heads sharing g (G*7 query rows), so a
// K/V tile crosses HBM once: one bulk copy (TMA) per tile into shared memory,
// used in place in the ring's own element type. The slot keys join the
// tile of rank 0. Scores and P.V are register-blocked over 4 / 2 query rows;
// each lane walks its key's 16-byte chunks in a lane-rotated order so that
// the 8 lanes of a quarter-warp touch distinct banks. Softmax is exp2-based
// in fp32. The partial (max, sum, O) of every CTA stays in its shared memory;
// after a cluster barrier, rank r combines rows r, r + nsplit, ... by reading
// all partners' partials through distributed shared memory in rank order
// (deterministic, no global round trip, no atomics).
//
// Memory read (same launch, CTAs of their own):
// y[s, h, p] = sum_n state[h, p, n] * C_s[s, n]. On the CUDA cores (fp32
// handles, other shapes) the state block of (b, h) is read with 16-byte
// loads, all in flight at once, and reduced across the lanes that share a
// state row; the bf16 form stages the heads by TMA and multiplies on the
// tensor cores (mem_tc_cta below). The state is never written here.
#include <mutex>

#include "common.cuh"

namespace hf {
namespace {

constexpr int MAXS = 16;     // max block slots
constexpr int THREADS = 256;
constexpr int MEM_QPT = 8;   // float4 state elements per thread (P*N <= 8192)
constexpr int MAX_SPLIT = 8; // portable cluster size

struct Plan {
  int nsplit;  // CTAs (cluster size) per (request, KV head)
  int jt;      // ring keys per CTA, multiple of 32
};

__host__ __device__ inline Plan make_plan(int W) {
  Plan p;
  p.nsplit = (W + 63) / 64;
  if (p.nsplit > MAX_SPLIT) p.nsplit = MAX_SPLIT;
  if (p.nsplit < 1) p.nsplit = 1;
  int per = (W + p.nsplit - 1) / p.nsplit;
  p.jt = (per + 31) / 32 * 32;
  return p;
}

struct Args {
  Dims d;
  Plan plan;
  int n_attn;     // attention CTAs = B * Hkv * nsplit
  int n_mem;      // memory-read CTAs = B * ceil(Hm / hpc)
  int hpc;        // memory heads per memory-read CTA
  int mem_first;  // tensor-core launch: 1 = memory-read CTAs before the attention CTAs
  int mem0;       // tensor-core launch: CTAs of the first kind, padded to whole clusters
  int mem_tc;     // 1: memory read on the tensor cores (tf32 mma.sync)
  int ntile;      // tensor-core path: 64-key window tiles per CTA
  float qscale;   // log2(e) / sqrt(dh)
  const float* proj;    // [B*S, Nd] fp32: Q | K_s | V_s | C_s
  const void* ring_k;   // [B][Hkv][W][dh] of this layer
  const void* ring_v;
  const int64_t* pos;   // [B]
  const float* state;   // [B][Hm][P][N] of this layer
  void* mix;            // [B*S, Nz]: O at columns [0, Hq*dh), y at [Hq*dh, Nz)
  int32_t* err;
  int early;      // what is final at launch (the previous launch signalled its
                  // dependents after its own dependency wait) and may be read before
                  // this launch's wait: EARLY_RING (ring K/V), EARLY_STATE (positions,
                  // states), EARLY_PROJ (the slot projections)
};

constexpr int EARLY_RING = 1, EARLY_STATE = 2, EARLY_PROJ = 4;

struct Layout {
  size_t bar, kt, vt, q, s, ml, total;
};

__host__ __device__ inline Layout make_layout(const Dims& d, const Plan& p, int esize) {
  Layout m{};
  size_t off = 0;
  const int R = d.G * d.S, JK = p.jt + d.S;
  m.bar = off;
  off += 16;
  m.kt = off;
  off += (size_t)JK * d.dh * esize;
  m.vt = off;
  off += (size_t)JK * d.dh * esize;
  m.q = off;  // query rows, later the partial O
  off += (size_t)R * (d.dh + 4) * 4;
  m.s = off;
  off += (size_t)R * JK * 4;
  m.ml = off;
  off += (size_t)R * 2 * 4;
  off = (off + 15) & ~(size_t)15;
  const size_t mem_need = (size_t)d.S * d.N * 4 + 16 * 4;  // C rows, 1/|C_s| (gated delta)
  m.total = off > mem_need ? off : mem_need;
  return m;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  return remote;
}
__device__ __forceinline__ float ld_peer_f(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// 16 bytes of T as floats.
template <typename T> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float* f) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <> struct Chunk<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float* f) {
    const float4 r = *reinterpret_cast<const float4*>(p);
    f[0] = r.x;
    f[1] = r.y;
    f[2] = r.z;
    f[3] = r.w;
  }
};

template <typename T, int E>
__device__ __forceinline__ void attn_cta(const Args& a, uint8_t* sm, int idx) {
  const Dims& d = a.d;
  const int nsplit = a.plan.nsplit, JT = a.plan.jt;
  const int rank = nsplit > 1 ? (int)cluster_rank() : 0;
  const int pair = idx / nsplit;
  const int kvh = pair % d.Hkv, b = pair / d.Hkv;
  const int S = d.S, G = d.G, R = G * S, dh = d.dh, dhp = dh + 4, JK = JT + S;
  constexpr int VE = Chunk<T>::N;
  const int nch = dh / VE;  // 16-byte chunks per key row
  const Layout L = make_layout(d, a.plan, (int)sizeof(T));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);
  T* kt = reinterpret_cast<T*>(sm + L.kt);
  T* vt = reinterpret_cast<T*>(sm + L.vt);
  float* q = reinterpret_cast<float*>(sm + L.q);
  float* s = reinterpret_cast<float*>(sm + L.s);
  float* ml = reinterpret_cast<float*>(sm + L.ml);
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid / 32, lane = tid % 32, nw = nthr / 32;

  pdl_wait();
  const long long p = __ldcg(&a.pos[b]);
  const int nv = (int)(p < (long long)d.W ? p : (long long)d.W);
  const int j0 = rank * JT;
  int nring = max(0, min(nv, j0 + JT) - j0);
  const int nslot = rank == 0 ? S : 0;
  const size_t rowbase = (size_t)b * S;
  const size_t rb = ((size_t)b * d.Hkv + kvh) * d.W * dh;

  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (nring > 0) {
      const uint32_t bytes = (uint32_t)(nring * dh * sizeof(T));
      mbar_expect_tx(bar, 2 * bytes);
      bulk_g2s(kt, static_cast<const T*>(a.ring_k) + rb + (size_t)j0 * dh, bytes, bar);
      bulk_g2s(vt, static_cast<const T*>(a.ring_v) + rb + (size_t)j0 * dh, bytes, bar);
    }
  }
  // Query rows (pre-scaled, fp32) and, on rank 0, the slot keys/values
  // appended after the ring tile in the ring's element type.
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
  if (nring > 0) ok = mbar_wait_for(bar, 0, d.wait);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      mbar_wait(bar, 0);  // bounded: let the copies land before the buffers are reused
    }
    nring = 0;  // drop the ring tile; the cluster sequence below stays matched
  }
  // slot keys/values go after the (possibly dropped) ring rows
  for (int i = tid; i < nslot * c4n; i += nthr) {
    const int j = i / c4n, c = (i % c4n) * 4;
    const float* row = a.proj + (rowbase + j) * d.Nd;
    const float4 kx = __ldcg(reinterpret_cast<const float4*>(row + d.QD + kvh * dh + c));
    const float4 vx = __ldcg(reinterpret_cast<const float4*>(row + d.QD + d.KVD + kvh * dh + c));
    T* kd = kt + (size_t)(nring + j) * dh + c;
    T* vd = vt + (size_t)(nring + j) * dh + c;
    kd[0] = from_f<T>(kx.x); kd[1] = from_f<T>(kx.y); kd[2] = from_f<T>(kx.z); kd[3] = from_f<T>(kx.w);
    vd[0] = from_f<T>(vx.x); vd[1] = from_f<T>(vx.y); vd[2] = from_f<T>(vx.z); vd[3] = from_f<T>(vx.w);
  }
  const int nk = nring + nslot;
  __syncthreads();

  // Scores: a half-warp takes one key, each of its 16 lanes a contiguous
  // slice of dh/16 elements (conflict-free); a warp owns 4 query rows whose
  // matching slices it keeps in registers across all keys. Partial dots are
  // summed over the 16 lanes of the half with shuffles.
  {
    const int half = lane / 16, hl = lane % 16;  // E = dh / 16 elements per lane
    const int rblocks = (R + 3) / 4;
    for (int rbk = warp; rbk < rblocks; rbk += nw) {
      const int r0 = rbk * 4;
      float qf[4][E];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = min(r0 + rr, R - 1);
#pragma unroll
        for (int e = 0; e < E; ++e) qf[rr][e] = q[r * dhp + hl * E + e];
      }
      for (int jp = 0; jp < nk; jp += 2) {
        const int j = jp + half;
        float kf[E];
        if (j < nk) {
          const T* kp = kt + (size_t)j * dh + hl * E;
          if constexpr (E == VE) {
            Chunk<T>::load(kp, kf);
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) kf[e] = to_f(kp[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) kf[e] = 0.f;
        }
        float acc[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          float a2 = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) a2 = fmaf(qf[rr][e], kf[e], a2);
          acc[rr] = a2;
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) acc[rr] += __shfl_xor_sync(0xffffffffu, acc[rr], o);
        if (hl == 0 && j < nk) {
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
            if (r0 + rr < R) {
              // cross-slot off: slot key j - nring counts for its own slot only
              const bool masked = d.xoff && j >= nring && j - nring != (r0 + rr) % S;
              s[(r0 + rr) * JK + j] = masked ? -INFINITY : acc[rr];
            }
        }
      }
    }
  }
  __syncthreads();

  // Softmax (unnormalised): one warp per row.
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
      ml[r * 2 + 0] = m;
      ml[r * 2 + 1] = l;
    }
  }
  __syncthreads();

  // P.V: item = (2 query rows, one 16-byte chunk of dh); the partial O
  // overwrites the query rows (no longer needed).
  {
    const int rblocks = (R + 1) / 2;
    float* o = q;
    for (int it = tid; it < rblocks * nch; it += nthr) {
      const int r0 = (it / nch) * 2, cc = it % nch;
      const int r1 = min(r0 + 1, R - 1);
      float acc0[VE], acc1[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) acc0[e] = acc1[e] = 0.f;
      for (int j = 0; j < nk; ++j) {
        float vf[VE];
        Chunk<T>::load(vt + (size_t)j * dh + cc * VE, vf);
        const float p0 = s[r0 * JK + j], p1 = s[r1 * JK + j];
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          acc0[e] = fmaf(p0, vf[e], acc0[e]);
          acc1[e] = fmaf(p1, vf[e], acc1[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < VE; e += 4) {
        *reinterpret_cast<float4*>(&o[r0 * dhp + cc * VE + e]) =
            make_float4(acc0[e], acc0[e + 1], acc0[e + 2], acc0[e + 3]);
        if (r0 + 1 < R)
          *reinterpret_cast<float4*>(&o[(r0 + 1) * dhp + cc * VE + e]) =
              make_float4(acc1[e], acc1[e + 1], acc1[e + 2], acc1[e + 3]);
      }
    }
  }

  T* mix = static_cast<T*>(a.mix);
  if (nsplit == 1) {
    __syncthreads();
    for (int i = tid; i < R * c4n; i += nthr) {
      const int r = i / c4n, c = (i % c4n) * 4, g = r / S, sl = r % S;
      const float inv = 1.f / ml[r * 2 + 1];
      const float4 x = *reinterpret_cast<const float4*>(&q[r * dhp + c]);
      T* dst = mix + (rowbase + sl) * d.Nz + (size_t)(kvh * G + g) * dh + c;
      dst[0] = from_f<T>(x.x * inv);
      dst[1] = from_f<T>(x.y * inv);
      dst[2] = from_f<T>(x.z * inv);
      dst[3] = from_f<T>(x.w * inv);
    }
    return;
  }

  // Combine through distributed shared memory: rank r owns rows r, r+nsplit, ...
  cluster_sync_all();
  const int my_rows = (R - rank + nsplit - 1) / nsplit;
  for (int i = tid; i < my_rows * c4n; i += nthr) {
    const int r = rank + (i / c4n) * nsplit, c = (i % c4n) * 4, g = r / S, sl = r % S;
    float mp[MAX_SPLIT], lp[MAX_SPLIT];
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < MAX_SPLIT; ++sp) {
      if (sp < nsplit) {
        const uint32_t ad = peer_addr(&ml[r * 2], (uint32_t)sp);
        mp[sp] = ld_peer_f(ad);
        lp[sp] = ld_peer_f(ad + 4);
        M = fmaxf(M, mp[sp]);
      }
    }
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < MAX_SPLIT; ++sp) {
      if (sp < nsplit) {
        const float wt = lp[sp] > 0.f ? exp2f(mp[sp] - M) : 0.f;
        const float4 ov = ld_peer_f4(peer_addr(&q[r * dhp + c], (uint32_t)sp));
        Lsum = fmaf(lp[sp], wt, Lsum);
        acc.x = fmaf(wt, ov.x, acc.x);
        acc.y = fmaf(wt, ov.y, acc.y);
        acc.z = fmaf(wt, ov.z, acc.z);
        acc.w = fmaf(wt, ov.w, acc.w);
      }
    }
    const float inv = 1.f / Lsum;
    T* dst = mix + (rowbase + sl) * d.Nz + (size_t)(kvh * G + g) * dh + c;
    dst[0] = from_f<T>(acc.x * inv);
    dst[1] = from_f<T>(acc.y * inv);
    dst[2] = from_f<T>(acc.z * inv);
    dst[3] = from_f<T>(acc.w * inv);
  }
  cluster_sync_all();  // partners keep their shared memory until every read is done
}

template <typename T>
__device__ __forceinline__ void mem_head(const Args& a, uint8_t* sm, int b, int hd) {
  const Dims& d = a.d;
  const int S = d.S, N = d.N, P = d.P;
  float* cs = reinterpret_cast<float*>(sm);
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid / 32, lane = tid % 32, nw = nthr / 32;
  pdl_wait();
  const float* hb = a.state + (((size_t)b * d.Hm + hd) * P) * N;
  T* mix = static_cast<T*>(a.mix);
  const int cC = d.QD + 2 * d.KVD;
  float* qn = cs + (size_t)S * N;  // gated delta: 1/|C_s|
  if (d.gdn) {
    __syncthreads();  // qn of the previous head fully consumed
    slot_inv_norms(a.proj + (size_t)b * S * d.Nd + cC, d.Nd, S, N, qn);
    __syncthreads();
  }
  if (N == 128 && S <= 8) {
    // lane l owns state columns 4l..4l+3; a warp takes 4 state rows at a time
    // and all slots: 4 x 8 partial dots per lane, one reduce-scatter.
    float4 c4[8];
#pragma unroll
    for (int sl = 0; sl < 8; ++sl)
      c4[sl] = sl < S ? __ldcg(reinterpret_cast<const float4*>(
                            a.proj + ((size_t)b * S + sl) * d.Nd + cC + 4 * lane))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = warp * 4; p0 < P; p0 += nw * 4) {
      float4 hv[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
        hv[rr] = p0 + rr < P ? __ldcg(reinterpret_cast<const float4*>(hb + (size_t)(p0 + rr) * N) + lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      float v[32];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int sl = 0; sl < 8; ++sl)
          v[rr * 8 + sl] = hv[rr].x * c4[sl].x + hv[rr].y * c4[sl].y + hv[rr].z * c4[sl].z +
                           hv[rr].w * c4[sl].w;
      const float tot = reduce_scatter32(v, lane);
      const int rr = lane / 8, sl = lane % 8, pr = p0 + rr;
      if (sl < S && pr < P)
        mix[((size_t)b * S + sl) * d.Nz + d.QD + (size_t)hd * P + pr] =
            from_f<T>(d.gdn ? tot * qn[sl] : tot);
    }
    return;
  }
  // general shapes: flat float4 walk, reduction across the lanes of a row
  const float4* h = reinterpret_cast<const float4*>(hb);
  const int nq = P * N / 4;
  __syncthreads();  // cs of the previous head fully consumed
  float4 hv[MEM_QPT];
#pragma unroll
  for (int u = 0; u < MEM_QPT; ++u) {
    const int qi = tid + u * nthr;
    hv[u] = qi < nq ? __ldcg(&h[qi]) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i = tid; i < S * N / 4; i += nthr) {
    const int sl = (i * 4) / N, n = (i * 4) % N;
    *reinterpret_cast<float4*>(&cs[sl * N + n]) =
        __ldcg(reinterpret_cast<const float4*>(a.proj + ((size_t)b * S + sl) * d.Nd + cC + n));
  }
  __syncthreads();
  const int gsz = N / 4;  // lanes sharing one state row (power of two <= 32)
#pragma unroll
  for (int u = 0; u < MEM_QPT; ++u) {
    if (u * nthr >= nq) break;  // uniform across the CTA
    const int qi = tid + u * nthr;
    const int pr = (qi * 4) / N, n = (qi * 4) % N;
#pragma unroll
    for (int sl = 0; sl < MAXS; ++sl) {
      if (sl >= S) break;
      const float4 c = *reinterpret_cast<const float4*>(&cs[sl * N + n]);
      float acc = hv[u].x * c.x + hv[u].y * c.y + hv[u].z * c.z + hv[u].w * c.w;
      for (int o = gsz / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if ((qi & (gsz - 1)) == 0 && qi < nq)
        mix[((size_t)b * S + sl) * d.Nz + d.QD + (size_t)hd * P + pr] =
            from_f<T>(d.gdn ? acc * qn[sl] : acc);
    }
  }
}

template <typename T>
__device__ __forceinline__ void mem_cta(const Args& a, uint8_t* sm, int idx) {
  const Dims& d = a.d;
  const int nhb = (d.Hm + a.hpc - 1) / a.hpc;
  const int b = idx / nhb, hd0 = (idx % nhb) * a.hpc;
  const int hd1 = min(d.Hm, hd0 + a.hpc);
  for (int hd = hd0; hd < hd1; ++hd) mem_head<T>(a, sm, b, hd);
}


// ---------------------------------------------------------------------------
// Tensor-core variant (bf16 rings, head_dim a multiple of 64): flash decoding.
//
// The valid part of the window of (request b, KV head g) is cut into tiles of
// KT = 64 keys; the nsplit CTAs of (b, g) (one cluster) take `ntile`
// consecutive tiles each, and rank 0 also takes the 7 slot keys: every tile
// buffer holds 64 ring rows (written by TMA) and 16 slot rows (written once
// by the threads), and rank 0's last tile covers all 80. The split count
// follows the batch: enough CTAs to fill the GPU at batch 1 (8 per cluster),
// one CTA per (b, g) walking the whole window at large batch. Ring tiles
// arrive by 2-D TMA through a TC_STAGES-deep ring of shared-memory buffers,
// in 128-byte-swizzled sub-tiles of 64 columns (16-byte chunk c of row r at
// chunk c ^ (r & 7)); Q (pre-scaled by log2(e)/sqrt(dh)) is written by the
// threads in the same layout, so every ldmatrix phase reads 8 distinct banks.
//
// Warp (m, k, h) owns query rows 16m..16m+15, the k-th group of KW keys of
// every tile and the h-th part of the head dimension of O. It runs its own
// flash-decoding loop: S = Q.K^T on mma.sync m16n8k16 (bf16 in, fp32
// accumulate; G*7 <= 64 query rows are below the 128-row minimum of the
// tcgen05 path), an online-softmax update of its row max m and sum l in
// registers (fp32, exp2), P rounded to bf16 and reused in registers as the
// A operand of O = scale * O + P.V (the row sums use the rounded values).
// Warps never wait on each other inside the loop; at the end the key groups
// are merged through shared memory, and a cluster merges its ranks' (m, l, O)
// through distributed shared memory in rank order.

constexpr int KT = 64;         // keys per window tile
constexpr int KTS = KT + 16;   // rows of a tile buffer: window tile + slot rows
constexpr int TC_STAGES = 2;   // window tiles in flight per CTA

// Warp roles of the tensor-core attention for a shape.
struct TcWarps {
  int mt, dp, kg, kw, dw;  // m-tiles, head-dim parts, key groups, keys / group, O columns / warp
};
__host__ __device__ inline TcWarps tc_warps(const Dims& d) {
  TcWarps w;
  w.mt = (d.G * d.S + 15) / 16;
  w.dp = d.dh > 128 ? d.dh / 128 : 1;
  w.kg = 8 / (w.mt * w.dp);
  if (w.kg > 4) w.kg = 4;
  if (w.kg < 1) w.kg = 1;
  w.kw = KT / w.kg;
  w.dw = d.dh / w.dp;
  return w;
}

struct TcLayout {
  size_t kv, okg, o, q, ml, mlk, bar, total;
  int qrows, stage;
};

__host__ __device__ inline TcLayout make_tc_layout(const Dims& d) {
  TcLayout m{};
  const TcWarps w = tc_warps(d);
  m.qrows = w.mt * 16;
  const int dsub = d.dh / 64;
  m.stage = dsub * KTS * 128;  // one K (or V) tile buffer, multiple of 1024 B
  size_t off = 0;
  // [stage][K | V]; after the last tile: the key groups' partial O, then the
  // CTA's partial O for the cluster combine
  m.kv = off;
  const size_t og = (size_t)w.kg * m.qrows * (d.dh + 4) * 4;
  const size_t o = (size_t)m.qrows * (d.dh + 4) * 4;
  size_t kv = (size_t)TC_STAGES * 2 * m.stage;
  if (og + o > kv) kv = og + o;
  kv = (kv + 1023) & ~(size_t)1023;
  m.okg = off;
  m.o = off + og;
  off += kv;
  m.q = off;
  off += (size_t)dsub * m.qrows * 128;
  m.ml = off;  // per row: the CTA's max and sum (cluster combine)
  off += (size_t)m.qrows * 2 * 4;
  m.mlk = off;  // per key group and row: max and sum
  off += (size_t)w.kg * m.qrows * 2 * 4;
  off = (off + 7) & ~(size_t)7;
  m.bar = off;
  off += TC_STAGES * 8;
  size_t mem_need = (size_t)d.S * d.N * 4 + 16 * 4;  // C rows, 1/|C_s| (gated delta)
  if (mem_tc_ok(d)) {
    const size_t t = mem_tc_bytes(d);
    if (t > mem_need) mem_need = t;
  }
  m.total = (off > mem_need ? off : mem_need) + 1024;  // + slack to 1024-align the base
  return m;
}

// Byte offset of 16-byte chunk c of row r in a swizzled tile of `rows` rows.
__device__ __forceinline__ uint32_t sw_chunk(int rows, int r, int c) {
  return (uint32_t)((c >> 3) * rows * 128 + r * 128 + ((((c & 7) ^ (r & 7))) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x on the special-function unit (ex2.approx.ftz; 2^-inf = 0). The
// probabilities it makes are rounded to bf16 right after, far coarser than
// its error.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A row's running max moves only when a chunk's max exceeds it by more than
// this (log2 units); otherwise the chunk's exponentials are taken against the
// older max and stay below 2^kRescaleLog2. (m, l, O) stay consistent either
// way, so the merges are unchanged and the result differs by rounding only.
constexpr float kRescaleLog2 = 8.f;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

template <int DH>
__device__ __forceinline__ void attn_tc_cta(const Args& a, const CUtensorMap* mk,
                                            const CUtensorMap* mv, uint8_t* sm_raw, int idx) {
  const Dims& d = a.d;
  const int nsplit = a.plan.nsplit;
  const int rank = nsplit > 1 ? (int)cluster_rank() : 0;
  const int pair = idx / nsplit;
  const int kvh = pair % d.Hkv, b = pair / d.Hkv;
  const int S = d.S, G = d.G, R = G * S;
  constexpr int dh = DH, dsub = DH / 64;
  constexpr int NTO = (DH > 128 ? 128 : DH) / 8;  // 16x8 O fragments per warp
  const TcLayout L = make_tc_layout(d);
  const TcWarps W = tc_warps(d);
  const int QR = L.qrows;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* kv = sm + L.kv;
  uint8_t* qt = sm + L.q;
  float* ml = reinterpret_cast<float*>(sm + L.ml);
  float* mlk = reinterpret_cast<float*>(sm + L.mlk);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid / 32, lane = tid % 32;
  const int g8 = lane >> 2, t4 = lane & 3;

  const bool ring_early = (a.early & EARLY_RING) != 0;
  const bool state_early = (a.early & EARLY_STATE) != 0;
  const int t0 = rank * a.ntile;
  const size_t rowbase = (size_t)b * S;
  const int y_head = (b * d.Hkv + kvh) * d.W;

  auto issue = [&](int i) {  // ring tile i of this CTA into its stage
    uint64_t* br = &bar[i % TC_STAGES];
    uint8_t* kd = kv + (size_t)(i % TC_STAGES) * 2 * L.stage;
    const int y0 = y_head + (t0 + i) * KT;
    mbar_expect_tx(br, (uint32_t)(2 * dsub * KT * 128));  // K and V, KT rows each
    for (int u = 0; u < dsub; ++u) {
      tma_load_2d(kd + (size_t)u * KTS * 128, mk, br, u * 64, y0);
      tma_load_2d(kd + L.stage + (size_t)u * KTS * 128, mv, br, u * 64, y0);
    }
  };
  auto init_bars = [&]() {
    for (int i = 0; i < TC_STAGES; ++i) mbar_init(&bar[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  };
  // Ring tiles requested before the valid count is known (ring final, the
  // positions not yet): the CTA's first tiles inside the window; those past
  // the valid rows are drained at the end.
  const bool proj_early = (a.early & EARLY_PROJ) != 0;
  const bool blind = ring_early && !state_early;
  const bool slots = rank == 0;
  bool waited = false;
  auto wait_once = [&]() {
    if (!waited) pdl_wait();
    waited = true;
  };
  constexpr int c4n = DH / 4;
  // Q rows (pre-scaled) as bf16, rows R..QR-1 zero; slot keys / values (rank
  // 0) into rows KT..KT+15 of every tile buffer (the copies write rows
  // 0..KT-1 only), rows past S zero (finite V for P.V). Each pass loads a
  // thread's QU Q pieces and SU slot pieces before it converts and stores any
  // of them, so a pass costs one L2 round trip (two passes at the serving
  // shape instead of a round trip per piece); a slot row is loaded once
  // for all tile buffers.
  constexpr int QU = 2, SU = 2;
  auto stage = [&]() {
    const int nq = QR * c4n, ns = slots ? 16 * c4n : 0;
    for (int pass = 0; pass * nthr * QU < nq || pass * nthr * SU < ns; ++pass) {
      float4 qx[QU], kx[SU], vx[SU];
#pragma unroll
      for (int u = 0; u < QU; ++u) {
        const int i = (pass * QU + u) * nthr + tid;
        const int r = i / c4n, c = (i % c4n) * 4;
        qx[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < nq && r < R)
          qx[u] = __ldcg(reinterpret_cast<const float4*>(
              a.proj + (rowbase + r % S) * d.Nd + (size_t)(kvh * G + r / S) * dh + c));
      }
#pragma unroll
      for (int u = 0; u < SU; ++u) {
        const int i = (pass * SU + u) * nthr + tid;
        const int j = i / c4n, c = (i % c4n) * 4;
        kx[u] = vx[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < ns && j < S) {
          const float* row = a.proj + (rowbase + j) * d.Nd;
          kx[u] = __ldcg(reinterpret_cast<const float4*>(row + d.QD + kvh * dh + c));
          vx[u] = __ldcg(reinterpret_cast<const float4*>(row + d.QD + d.KVD + kvh * dh + c));
        }
      }
#pragma unroll
      for (int u = 0; u < QU; ++u) {
        const int i = (pass * QU + u) * nthr + tid;
        if (i < nq) {
          const int r = i / c4n, c = (i % c4n) * 4;
          const float4 x = qx[u];
          *reinterpret_cast<uint2*>(qt + sw_chunk(QR, r, c >> 3) + (c & 7) * 2) =
              make_uint2(pack_bf16x2(x.x * a.qscale, x.y * a.qscale),
                         pack_bf16x2(x.z * a.qscale, x.w * a.qscale));
        }
      }
#pragma unroll
      for (int u = 0; u < SU; ++u) {
        const int i = (pass * SU + u) * nthr + tid;
        if (i < ns) {
          const int j = i / c4n, c = (i % c4n) * 4;
          const uint2 kw = make_uint2(pack_bf16x2(kx[u].x, kx[u].y), pack_bf16x2(kx[u].z, kx[u].w));
          const uint2 vw = make_uint2(pack_bf16x2(vx[u].x, vx[u].y), pack_bf16x2(vx[u].z, vx[u].w));
          const uint32_t off = sw_chunk(KTS, KT + j, c >> 3) + (c & 7) * 2;
#pragma unroll
          for (int stg = 0; stg < TC_STAGES; ++stg) {
            uint8_t* kd = kv + (size_t)stg * 2 * L.stage;
            *reinterpret_cast<uint2*>(kd + off) = kw;
            *reinterpret_cast<uint2*>(kd + L.stage + off) = vw;
          }
        }
      }
    }
  };
  int nissue = 0;
  if (blind) {
    nissue = min(TC_STAGES, min(a.ntile, (d.W + KT - 1) / KT - t0));
    if (tid == 0) {
      init_bars();
      for (int i = 0; i < nissue; ++i) issue(i);
    }
  }
  if (proj_early) stage();
  if (!state_early) wait_once();
  const long long p = __ldcg(&a.pos[b]);
  const int nv = (int)(p < (long long)d.W ? p : (long long)d.W);  // valid ring rows 0..nv-1
  const int nwt = max(0, min(a.ntile, (nv + KT - 1) / KT - t0));  // ring tiles of this CTA
  const int nsteps = max(nwt, slots ? 1 : 0);
  if (!blind) {
    if (!ring_early) wait_once();
    nissue = min(TC_STAGES, nwt);
    if (tid == 0) {
      init_bars();
      for (int i = 0; i < nissue; ++i) issue(i);
    }
  }
  if (!proj_early) {
    wait_once();  // the projections come from the previous launch
    stage();
  }
  __syncthreads();  // barriers initialised, Q and slot rows written

  // this warp's role
  const int nact = W.mt * W.kg * W.dp;
  const bool active = warp < nact;
  const int wdp = warp % W.dp, wkg = (warp / W.dp) % W.kg, wmt = warp / (W.dp * W.kg);
  float o[NTO][4];
#pragma unroll
  for (int k = 0; k < NTO; ++k) o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max of rows g8, g8 + 8 of the m-tile
  float l0 = 0.f, l1 = 0.f;              // this lane's part of the running sums
  const int qrow = wmt * 16 + (lane & 15);
  // ldmatrix addresses: a fragment's 16-byte chunk index within its 128-byte
  // row is (2 * step + half) XOR (row & 7); the half bit and the row phase are
  // per lane, the step is a compile-time constant
  const uint32_t qbase = smem_u32(qt) + (uint32_t)qrow * 128;
  const uint32_t qblk = (uint32_t)QR * 128;                              // one 64-column block of Q
  const uint32_t qh4 = (uint32_t)(((lane >> 4) ^ (lane & 7)) << 4);       // Q and V rows
  const uint32_t kh4 = (uint32_t)((((lane >> 3) & 1) ^ (lane & 7)) << 4);  // K rows
  const uint32_t vcol = (uint32_t)(wdp * (NTO / 8)) * KTS * 128;          // this warp's V columns

  // slots of this lane's two rows (cross-slot off masks the other slots' keys)
  const int sl0 = (wmt * 16 + g8) % S, sl1 = (wmt * 16 + g8 + 8) % S;

  // One online-softmax update over the 16 keys at tile rows kr..kr+15 of the
  // K/V buffers kb/vb; key row j is valid when j < lim (and, for the slot
  // keys with cross-slot attention off, when it is the row's own slot).
  auto update = [&](uint32_t kb, uint32_t vb, int kr, int lim) {
    const bool own_slot = d.xoff && kr >= KT;
    // [n-fragment][k-step parity][...]: two shorter mma chains per fragment
    // (one at head dim 256, where the registers are needed for O)
    constexpr int CH = DH > 128 ? 1 : 2;
    float sc[2][CH][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int h = 0; h < CH; ++h) sc[n][h][0] = sc[n][h][1] = sc[n][h][2] = sc[n][h][3] = 0.f;
    // S = Q K^T: per k-step one Q fragment and one K fragment pair
    const uint32_t krow = kb + (uint32_t)(kr + (lane & 7) + ((lane >> 4) << 3)) * 128;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      const uint32_t ph = (uint32_t)((ks & 3) << 5);
      ldsm_x4(qbase + (uint32_t)(ks >> 2) * qblk + (ph ^ qh4), a0, a1, a2, a3);
      ldsm_x4(krow + (uint32_t)((ks >> 2) * KTS * 128) + (ph ^ kh4), b0, b1, b2, b3);
      mma_bf16_16816(sc[0][ks % CH], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(sc[1][ks % CH], a0, a1, a2, a3, b2, b3);
    }
    float x0 = -INFINITY, x1 = -INFINITY;  // masked row maxima (quad of lanes per row)
    float t[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const int j = kr + n * 8 + 2 * t4;
#pragma unroll
      for (int e = 0; e < 4; ++e) t[n][e] = CH == 2 ? sc[n][0][e] + sc[n][CH - 1][e] : sc[n][0][e];
      if (j >= lim) t[n][0] = t[n][2] = -INFINITY;
      if (j + 1 >= lim) t[n][1] = t[n][3] = -INFINITY;
      if (own_slot) {  // cross-slot off: a slot key counts for its own slot's rows only
        const int js = j - KT;
        if (js != sl0) t[n][0] = -INFINITY;
        if (js + 1 != sl0) t[n][1] = -INFINITY;
        if (js != sl1) t[n][2] = -INFINITY;
        if (js + 1 != sl1) t[n][3] = -INFINITY;
      }
      x0 = fmaxf(x0, fmaxf(t[n][0], t[n][1]));
      x1 = fmaxf(x1, fmaxf(t[n][2], t[n][3]));
    }
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
    if (__any_sync(0xffffffffu, x0 > m0 + kRescaleLog2 || x1 > m1 + kRescaleLog2)) {
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      const float s0 = n0 == -INFINITY ? 1.f : ex2_fast(m0 - n0);
      const float s1 = n1 == -INFINITY ? 1.f : ex2_fast(m1 - n1);
      m0 = n0;
      m1 = n1;
      l0 *= s0;
      l1 *= s1;
#pragma unroll
      for (int k = 0; k < NTO; ++k) {
        o[k][0] *= s0;
        o[k][1] *= s0;
        o[k][2] *= s1;
        o[k][3] *= s1;
      }
    }
    // P = exp2(S - m) rounded to bf16, packed as the A operand of P.V
    uint32_t pa[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      pa[n][0] = pack_bf16x2(ex2_fast(t[n][0] - m0), ex2_fast(t[n][1] - m0));
      pa[n][1] = pack_bf16x2(ex2_fast(t[n][2] - m1), ex2_fast(t[n][3] - m1));
      const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa[n][0]));
      const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa[n][1]));
      l0 += r0.x + r0.y;
      l1 += r1.x + r1.y;
    }
    // O += P V over this warp's head-dim part, two 8-column fragments per load
    const int key = kr + (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t vrow = vb + (uint32_t)key * 128 + vcol;
#pragma unroll
    for (int k = 0; k < NTO; k += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vrow + (uint32_t)((k >> 3) * KTS * 128) + ((uint32_t)((k & 7) << 4) ^ qh4), b0,
                b1, b2, b3);
      mma_bf16_16816(o[k], pa[0][0], pa[0][1], pa[1][0], pa[1][1], b0, b1);
      mma_bf16_16816(o[k + 1], pa[0][0], pa[0][1], pa[1][0], pa[1][1], b2, b3);
    }
  };

  int done = 0;  // ring tiles consumed
  bool aborted = false;
  for (int i = 0; i < nsteps; ++i) {
    const bool ring = i < nwt;  // a window tile arrives in stage i % STAGES
    const bool with_slots = slots && i == nsteps - 1;
    const int nvr = ring ? min(KT, nv - (t0 + i) * KT) : 0;  // valid window rows
    uint8_t* kt = kv + (size_t)(ring ? i % TC_STAGES : 0) * 2 * L.stage;
    uint8_t* vt = kt + L.stage;
    if (ring) {
      const bool ok = mbar_wait(&bar[i % TC_STAGES], (uint32_t)((i / TC_STAGES) & 1));
      if (!__syncthreads_and(ok)) {
        aborted = true;
        break;
      }
      // window rows past the valid ones: V zeroed (P is zero there, V must be finite)
      if (nvr < KT) {
        for (int e = tid; e < (KT - nvr) * c4n; e += nthr) {
          const int j = nvr + e / c4n, c = (e % c4n) * 4;
          *reinterpret_cast<uint2*>(vt + sw_chunk(KTS, j, c >> 3) + (c & 7) * 2) =
              make_uint2(0u, 0u);
        }
        __syncthreads();
      }
      done = i + 1;
    }
    if (active && ring)
      for (int q = 0; q < W.kw; q += 16)
        if (wkg * W.kw + q < nvr) update(smem_u32(kt), smem_u32(vt), wkg * W.kw + q, nvr);
    // the slot keys (rows KT..KT+15) go to the last key group
    if (with_slots && active && wkg == W.kg - 1)
      update(smem_u32(kt), smem_u32(vt), KT, KT + S);
    if (ring) {
      __syncthreads();  // every warp done with this stage
      if (tid == 0 && i + TC_STAGES < nwt) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(i + TC_STAGES);
      }
    }
  }

  if (aborted) {
    // a tile copy never completed: report, let the copies in flight land
    // (bounded) before the shared memory is released, write nothing
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      const int issued = max(nissue, min(nwt, done + TC_STAGES));
      for (int i = done; i < issued; ++i)
        mbar_wait(&bar[i % TC_STAGES], (uint32_t)((i / TC_STAGES) & 1));
    }
    if (nsplit > 1) {
      cluster_sync_all();  // matches the two cluster barriers of the combine
      cluster_sync_all();
    }
    return;
  }

  // tiles requested past the valid rows: let their copies land first
  if (tid == 0)
    for (int i = nwt; i < nissue; ++i) mbar_wait(&bar[i % TC_STAGES], (uint32_t)((i / TC_STAGES) & 1));
  // key groups -> shared memory (the tile buffers are free now)
  __syncthreads();
  float* okg = reinterpret_cast<float*>(sm + L.okg);  // [kg][QR][dh + 4]
  float* octa = reinterpret_cast<float*>(sm + L.o);   // [QR][dh + 4]
  const int OLD = dh + 4;
  if (active) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int r = wmt * 16 + g8;
    float* ob = okg + ((size_t)wkg * QR + r) * OLD + wdp * W.dw + 2 * t4;
#pragma unroll
    for (int k = 0; k < NTO; ++k) {
      *reinterpret_cast<float2*>(ob + k * 8) = make_float2(o[k][0], o[k][1]);
      *reinterpret_cast<float2*>(ob + 8 * OLD + k * 8) = make_float2(o[k][2], o[k][3]);
    }
    if (t4 == 0 && wdp == 0) {
      float* mb = mlk + ((size_t)wkg * QR + r) * 2;
      mb[0] = m0;
      mb[1] = l0;
      mb[16] = m1;
      mb[17] = l1;
    }
  }
  __syncthreads();
  __nv_bfloat16* mix = static_cast<__nv_bfloat16*>(a.mix);
  const int c = (tid % c4n) * 4, rstep = nthr / c4n;
  if (nsplit == 1) {
    // merge the key groups per row and write O: every thread of a row forms
    // the groups' weights w_k = 2^(m_k - M) itself (M = max m_k), then sums
    // its 4 columns: O = sum w_k O_k / sum w_k l_k
    for (int r = tid / c4n; r < R; r += rstep) {
      float mk[4], lk[4];
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mk[k] = k < W.kg ? mlk[((size_t)k * QR + r) * 2] : -INFINITY;
        lk[k] = k < W.kg ? mlk[((size_t)k * QR + r) * 2 + 1] : 0.f;
        M = fmaxf(M, mk[k]);
      }
      float Ls = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (k >= W.kg) break;
        const float wt = lk[k] > 0.f ? ex2_fast(mk[k] - M) : 0.f;  // an empty group weighs 0
        Ls = fmaf(wt, lk[k], Ls);
        const float4 ov = *reinterpret_cast<const float4*>(okg + ((size_t)k * QR + r) * OLD + c);
        acc.x = fmaf(wt, ov.x, acc.x);
        acc.y = fmaf(wt, ov.y, acc.y);
        acc.z = fmaf(wt, ov.z, acc.z);
        acc.w = fmaf(wt, ov.w, acc.w);
      }
      const float inv = 1.f / Ls;
      const int g = r / S, sl = r % S;
      __nv_bfloat16* dst = mix + (rowbase + sl) * d.Nz + (size_t)(kvh * G + g) * dh + c;
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    return;
  }
  // several ranks: merge the key groups per row: M = max m_k, L = sum w_k l_k,
  // O = sum w_k O_k. First one thread per row turns each group's max into its
  // weight w_k (in place) and keeps L with M.
  for (int r = tid; r < R; r += nthr) {
    float M = -INFINITY;
    for (int k = 0; k < W.kg; ++k) M = fmaxf(M, mlk[((size_t)k * QR + r) * 2]);
    float Ls = 0.f;
    for (int k = 0; k < W.kg; ++k) {
      float* e = mlk + ((size_t)k * QR + r) * 2;
      const float lk = e[1];
      const float wt = lk > 0.f ? ex2_fast(e[0] - M) : 0.f;  // an empty group weighs 0
      Ls = fmaf(wt, lk, Ls);
      e[0] = wt;
    }
    ml[r * 2] = M;
    ml[r * 2 + 1] = Ls;
  }
  __syncthreads();
  // then thread tid sums 4 columns (c) of rows r0, r0 + rstep, ...
  for (int r = tid / c4n; r < R; r += rstep) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < W.kg; ++k) {
      const float wt = mlk[((size_t)k * QR + r) * 2];
      const float4 ov = *reinterpret_cast<const float4*>(okg + ((size_t)k * QR + r) * OLD + c);
      acc.x = fmaf(wt, ov.x, acc.x);
      acc.y = fmaf(wt, ov.y, acc.y);
      acc.z = fmaf(wt, ov.z, acc.z);
      acc.w = fmaf(wt, ov.w, acc.w);
    }
    *reinterpret_cast<float4*>(octa + (size_t)r * OLD + c) = acc;
  }
  cluster_sync_all();
  // rank `rank` combines rows rank, rank + nsplit, ... over all ranks; every
  // partner's (m, l, O) is requested at once (one round trip)
  for (int r = rank + (tid / c4n) * nsplit; r < R; r += rstep * nsplit) {
    const int g = r / S, sl = r % S;
    float mp[MAX_SPLIT], lp[MAX_SPLIT];
    float4 op[MAX_SPLIT];
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < MAX_SPLIT; ++sp) {
      if (sp < nsplit) {
        const uint32_t ad = peer_addr(&ml[r * 2], (uint32_t)sp);
        mp[sp] = ld_peer_f(ad);
        lp[sp] = ld_peer_f(ad + 4);
        op[sp] = ld_peer_f4(peer_addr(octa + (size_t)r * OLD + c, (uint32_t)sp));
      }
    }
#pragma unroll
    for (int sp = 0; sp < MAX_SPLIT; ++sp)
      if (sp < nsplit) M = fmaxf(M, mp[sp]);
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < MAX_SPLIT; ++sp) {
      if (sp < nsplit) {
        const float wt = lp[sp] > 0.f ? exp2f(mp[sp] - M) : 0.f;
        const float4 ov = op[sp];
        Lsum = fmaf(lp[sp], wt, Lsum);
        acc.x = fmaf(wt, ov.x, acc.x);
        acc.y = fmaf(wt, ov.y, acc.y);
        acc.z = fmaf(wt, ov.z, acc.z);
        acc.w = fmaf(wt, ov.w, acc.w);
      }
    }
    const float inv = 1.f / Lsum;
    __nv_bfloat16* dst = mix + (rowbase + sl) * d.Nz + (size_t)(kvh * G + g) * dh + c;
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  }
  cluster_sync_all();  // partners keep their shared memory until every read is done
}

// Memory read CTA (tensor-core form, see common.cuh) over its heads: each
// head's state (P x N fp32) arrives by TMA in one of MEM_NBUF shared-memory
// buffers, MEM_NBUF - 1 heads ahead of the one being read, as 128-byte
// column groups of P rows in the 128-byte swizzle (16-byte chunk c of row r
// at chunk c ^ (r & 7)), so that the fragment loads below are conflict-free.
// Warp (m-tile, k-part) reads its 16 rows x (N / parts) columns from the
// buffer and multiplies them with the C rows on mma.sync (tf32); the k-parts
// are summed through shared memory. Every wait is bounded; on expiry the CTA
// raises ERR_TIMEOUT, lets the copies it issued land (bounded) and returns.
__device__ __forceinline__ void mem_tc_cta(const Args& a, const CUtensorMap* ms, uint8_t* sm_raw,
                                           int idx) {
  const Dims& d = a.d;
  const int nhb = (d.Hm + a.hpc - 1) / a.hpc;
  const int b = idx / nhb, hd0 = (idx % nhb) * a.hpc;
  const int nh = min(d.Hm, hd0 + a.hpc) - hd0;
  const int P = d.P, N = d.N, S = d.S;
  const int MT = P / 16, KSPL = mem_ksplit(d), G16 = N / 16 / KSPL;
  const size_t SB = mem_stage_bytes(d);
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sbuf = sm;                                                   // [MEM_NBUF][groups][P][128 B]
  float* red = reinterpret_cast<float*>(sm + MEM_NBUF * SB);          // [KSPL][P][8]
  float* qn = red + (size_t)KSPL * P * 8;                              // gated delta: 1/|C_s|
  uint64_t* bar = reinterpret_cast<uint64_t*>(qn + 16);               // [MEM_NBUF]
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int mt = warp % MT, kp = warp / MT;
  const bool active = kp < KSPL;
  const int r0 = mt * 16 + g8;
  const int col0 = kp * G16 * 16 + 4 * t4;  // this lane's first column
  const bool state_early = (a.early & EARLY_STATE) != 0;
  const int ngroups = (N + 31) / 32;
  const int y0 = (b * d.Hm + hd0) * P;  // first state row of this CTA's heads
  auto issue = [&](int i) {  // head i into buffer i % MEM_NBUF (thread 0)
    uint8_t* dst = sbuf + (size_t)(i % MEM_NBUF) * SB;
    uint64_t* br = &bar[i % MEM_NBUF];
    mbar_expect_tx(br, (uint32_t)SB);
    for (int g = 0; g < ngroups; ++g)
      tma_load_2d(dst + (size_t)g * P * 128, ms, br, g * 32, y0 + i * P);
  };
  const int pre = nh < MEM_NBUF - 1 ? nh : MEM_NBUF - 1;
  if (tid == 0) {
    for (int k = 0; k < MEM_NBUF; ++k) mbar_init(&bar[k], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (!state_early) pdl_wait();
  if (tid == 0)
    for (int i = 0; i < pre; ++i) issue(i);
  if (state_early) pdl_wait();  // C comes from the previous launch
  // B fragments (C of this request, slot g8), held for all heads
  uint32_t bf[MEM_G16][4];
  {
    const float* crow = a.proj + ((size_t)b * S + g8) * d.Nd + d.QD + 2 * d.KVD + col0;
#pragma unroll
    for (int j = 0; j < MEM_G16; ++j) {
      float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && j < G16 && g8 < S) c = __ldcg(reinterpret_cast<const float4*>(crow + j * 16));
      bf[j][0] = to_tf32(c.x);
      bf[j][1] = to_tf32(c.y);
      bf[j][2] = to_tf32(c.z);
      bf[j][3] = to_tf32(c.w);
    }
  }
  if (d.gdn) slot_inv_norms(a.proj + (size_t)b * S * d.Nd + d.QD + 2 * d.KVD, d.Nd, S, N, qn);
  __nv_bfloat16* mix = static_cast<__nv_bfloat16*>(a.mix);
  int issued = pre, done = 0;
  bool ok = true;
  for (int i = 0; i < nh; ++i) {
    // the buffer of head i + MEM_NBUF - 1 held head i - 1, read by every warp
    // before the barrier after its partial sums
    if (tid == 0 && issued < nh && issued == i + MEM_NBUF - 1) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(issued++);
    }
    ok = mbar_wait(&bar[i % MEM_NBUF], (uint32_t)((i / MEM_NBUF) & 1));
    if (!__syncthreads_and(ok)) break;  // and the previous head's sums are read
    done = i + 1;
    if (active) {
      const uint8_t* hs = sbuf + (size_t)(i % MEM_NBUF) * SB;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < MEM_G16; ++j)
        if (j < G16) {
          const int col = col0 + j * 16;  // 4 columns: one 16-byte chunk of a 128-byte group
          const uint8_t* gb = hs + (size_t)(col >> 5) * P * 128;
          const int ch = (col & 31) >> 2;
          const float4 h0 = *reinterpret_cast<const float4*>(gb + r0 * 128 + ((ch ^ (r0 & 7)) << 4));
          const float4 h1 =
              *reinterpret_cast<const float4*>(gb + (r0 + 8) * 128 + ((ch ^ ((r0 + 8) & 7)) << 4));
          mma_tf32_1688(c, to_tf32(h0.x), to_tf32(h1.x), to_tf32(h0.y), to_tf32(h1.y), bf[j][0],
                        bf[j][1]);
          mma_tf32_1688(c, to_tf32(h0.z), to_tf32(h1.z), to_tf32(h0.w), to_tf32(h1.w), bf[j][2],
                        bf[j][3]);
        }
      // c: (row r0, slots 2t4, 2t4+1), (row r0 + 8, same slots)
      float* rp = red + ((size_t)kp * P + r0) * 8 + 2 * t4;
      *reinterpret_cast<float2*>(rp) = make_float2(c[0], c[1]);
      *reinterpret_cast<float2*>(rp + 64) = make_float2(c[2], c[3]);
    }
    __syncthreads();
    for (int e = tid; e < S * P; e += blockDim.x) {
      const int sl = e / P, p = e % P;
      float y = 0.f;
      for (int q = 0; q < KSPL; ++q) y += red[((size_t)q * P + p) * 8 + sl];
      if (d.gdn) y *= qn[sl];
      mix[((size_t)b * S + sl) * d.Nz + d.QD + (size_t)(hd0 + i) * P + p] = __float2bfloat16_rn(y);
    }
  }
  if (!ok && tid == 0) {
    // a copy never completed: report, and let the copies in flight land
    // (bounded) before the shared memory is released
    atomicOr(a.err, ERR_TIMEOUT);
    for (int i = done; i < issued; ++i) mbar_wait(&bar[i % MEM_NBUF], (uint32_t)((i / MEM_NBUF) & 1));
  }
}

template <int DH>
__global__ void __launch_bounds__(THREADS, 2)
attn_tc_kernel(Args a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
               const __grid_constant__ CUtensorMap ms) {
  extern __shared__ __align__(128) uint8_t sm[];
  pdl_trigger();
  // launches of more than one wave: the memory-read CTAs first (few,
  // long-lived), then the attention CTAs (many, short: they pack the
  // launch's tail); a single wave: the attention CTAs (the critical path)
  // first. Each kind starts on a whole cluster.
  const int idx = blockIdx.x;
  const int att0 = a.mem_first ? a.mem0 : 0;  // first attention CTA
  const int mem0 = a.mem_first ? 0 : a.mem0;  // first memory-read CTA
  if (idx >= att0 && idx - att0 < a.n_attn) {
    attn_tc_cta<DH>(a, &mk, &mv, sm, idx - att0);
  } else if (idx >= mem0 && idx - mem0 < a.n_mem) {
    if (a.mem_tc)
      mem_tc_cta(a, &ms, sm, idx - mem0);
    else
      mem_cta<__nv_bfloat16>(a, sm, idx - mem0);
  } else {
    pdl_wait();  // cluster padding
  }
}

// E = head_dim / 16: the slice of a key each lane of a half-warp holds.
template <typename T, int E>
__global__ void __launch_bounds__(THREADS) attn_cluster_kernel(Args a) {
  extern __shared__ __align__(128) uint8_t sm[];
  pdl_trigger();
  const int idx = blockIdx.x;
  if (idx < a.n_attn)
    attn_cta<T, E>(a, sm, idx);
  else if (idx < a.n_attn + a.n_mem)
    mem_cta<T>(a, sm, idx - a.n_attn);
  else
    pdl_wait();  // cluster padding
}

}  // namespace

bool attn_uses_tc(const Dims& d, int dtype) {
  const int qrows = (d.G * d.S + 15) / 16 * 16;
  // the warp roles need m-tiles x head-dim parts <= 4 (at least two key groups)
  return dtype == HF_BF16 && d.dh % 64 == 0 && qrows * d.dh <= 8192;
}

int attn_tile_rows(const Dims&) { return KT; }

size_t attn_cluster_smem(const Dims& d, int esize) {
  if (esize == 2 && attn_uses_tc(d, HF_BF16)) return make_tc_layout(d).total;
  return make_layout(d, make_plan(d.W), esize).total;
}

constexpr int kMaxSmem = 232448;  // opt-in shared memory per CTA

template <typename K>
cudaError_t configure_kernel(K kernel) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

template <typename T>
cudaError_t configure_dtype() {
  cudaError_t e = configure_kernel(attn_cluster_kernel<T, 2>);
  if (e == cudaSuccess) e = configure_kernel(attn_cluster_kernel<T, 4>);
  if (e == cudaSuccess) e = configure_kernel(attn_cluster_kernel<T, 8>);
  if (e == cudaSuccess) e = configure_kernel(attn_cluster_kernel<T, 16>);
  return e;
}

// Every variant may use up to the opt-in maximum; the launch passes the
// layout's own size, which sets the occupancy.
// (The attributes are per-device settings: configured once per device.)
cudaError_t configure_attn_cluster(const Dims&) {
  constexpr int kMaxDevices = 64;
  static bool configured[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (configured[dev]) return cudaSuccess;
  e = configure_dtype<float>();
  if (e == cudaSuccess) e = configure_dtype<__nv_bfloat16>();
  if (e == cudaSuccess) e = configure_kernel(attn_tc_kernel<64>);
  if (e == cudaSuccess) e = configure_kernel(attn_tc_kernel<128>);
  if (e == cudaSuccess) e = configure_kernel(attn_tc_kernel<256>);
  if (e == cudaSuccess) configured[dev] = true;
  return e;
}

template <typename T>
cudaError_t launch_typed(const cudaLaunchConfig_t& cfg, const Args& a) {
  switch (a.d.dh) {
    case 32: return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<T, 2>, a);
    case 64: return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<T, 4>, a);
    case 128: return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<T, 8>, a);
    case 256: return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<T, 16>, a);
  }
  return cudaErrorInvalidValue;
}

// Split of the tensor-core path: about two CTAs per SM over the batch's
// (request, KV head) pairs, at most 8 (one cluster) and no more than the
// window has tiles; every rank gets the same number of tiles.
static Plan make_tc_plan(const Dims& d, int B, int num_sms, int* ntile) {
  const int nwin = (d.W + KT - 1) / KT;
  const int pairs = B * d.Hkv;
  int ns = (2 * num_sms + pairs - 1) / pairs;
  ns = ns < 1 ? 1 : (ns > MAX_SPLIT ? MAX_SPLIT : ns);
  if (ns > nwin) ns = nwin;
  *ntile = (nwin + ns - 1) / ns;
  Plan p;
  p.nsplit = (nwin + *ntile - 1) / *ntile;
  p.jt = *ntile * KT;
  return p;
}

cudaError_t launch_attn_cluster(int dtype, const Dims& d, int B, const float* proj,
                                const void* ring_k, const void* ring_v, const int64_t* pos,
                                const float* state, void* mix, const CUtensorMap* mk,
                                const CUtensorMap* mv, const CUtensorMap* ms, int32_t* err,
                                int num_sms, int early, int with_mem, cudaStream_t st,
                                int* launches) {
  if (B <= 0) return cudaSuccess;
  const bool tc = attn_uses_tc(d, dtype) && mk && mv;
  Args a{};
  a.d = d;
  if (tc)
    a.plan = make_tc_plan(d, B, num_sms, &a.ntile);
  else
    a.plan = make_plan(d.W);
  a.n_attn = B * d.Hkv * a.plan.nsplit;
  a.mem_tc = tc && mem_tc_ok(d) && ms ? 1 : 0;
  if (a.mem_tc) {
    // staged memory reads (their copies pipelined over the CTA's heads): about
    // two long-lived CTAs per SM in all
    const int per_req = std::max(1, 2 * num_sms / B);
    a.hpc = (d.Hm + per_req - 1) / per_req;
  } else {
    // memory-read CTAs: one head each up to ~8 CTAs per SM, then several
    a.hpc = (B * d.Hm + 8 * num_sms - 1) / (8 * num_sms);
  }
  if (a.hpc < 1) a.hpc = 1;
  a.n_mem = with_mem ? B * ((d.Hm + a.hpc - 1) / a.hpc) : 0;
  a.qscale = 1.4426950408889634f / sqrtf((float)d.dh);
  a.proj = proj;
  a.ring_k = ring_k;
  a.ring_v = ring_v;
  a.pos = pos;
  a.state = state;
  a.mix = mix;
  a.err = err;
  a.early = tc ? early : 0;
  const int cz = a.plan.nsplit;
  const int mem_pad = (a.n_mem + cz - 1) / cz * cz, attn_pad = (a.n_attn + cz - 1) / cz * cz;
  a.mem_first = tc && a.n_attn + a.n_mem > 2 * num_sms ? 1 : 0;
  a.mem0 = a.mem_first ? mem_pad : attn_pad;
  const int total = tc ? mem_pad + attn_pad : (a.n_attn + a.n_mem + cz - 1) / cz * cz;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(total);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = tc ? make_tc_layout(d).total
                            : make_layout(d, a.plan, dtype == HF_F32 ? 4 : 2).total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cz;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  ++*launches;
  if (tc) {
    switch (d.dh) {
      // (without a state map the memory-read CTAs take the CUDA-core form and
      // the map argument is not read)
      case 64: return cudaLaunchKernelEx(&cfg, attn_tc_kernel<64>, a, *mk, *mv, ms ? *ms : *mk);
      case 128: return cudaLaunchKernelEx(&cfg, attn_tc_kernel<128>, a, *mk, *mv, ms ? *ms : *mk);
      case 256: return cudaLaunchKernelEx(&cfg, attn_tc_kernel<256>, a, *mk, *mv, ms ? *ms : *mk);
    }
    return cudaErrorInvalidValue;
  }
  if (dtype == HF_F32) return launch_typed<float>(cfg, a);
  return launch_typed<__nv_bfloat16>(cfg, a);
}

}  // namespace hf
