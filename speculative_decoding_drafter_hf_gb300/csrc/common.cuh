// Shared device helpers and the internal (non-ABI) interface between the
// runtime (hyflash.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "hyflash.h"

namespace hf {

// ---------------------------------------------------------------- dtype glue
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Stable softplus in fp32: max(x,0) + log1p(exp(-|x|)).
__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

// Logistic function (gated-delta writing strength).
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: every kernel of a round lets the next one
// start as soon as all of its CTAs are running (launch_dependents), and waits
// for the previous kernel's completion and memory (wait) before it reads or
// writes anything that kernel may touch. Every kernel calls pdl_wait before it
// finishes, so completion stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------- mbarrier / bulk copy
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz: bound of every wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete within `limit` clock
// cycles; false on timeout. A limit of 0 gives up before the first poll (its
// deadline has already passed): the hook the failure-detection tests use to
// run a kernel's expiry path without any copy going missing.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, long long limit) {
  if (limit <= 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

// Bounded wait with the default limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitCycles);
}

// 1-D bulk copy global -> shared (addresses 16-byte aligned, bytes % 16 == 0),
// completing `bytes` of transaction on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled TMA load (tensor map in param/const/global space) completing on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Device error word bits.
enum : int32_t { ERR_BAD_ACCEPTED = 1, ERR_TIMEOUT = 2 };

// ---------------------------------------------------------------- dims
// All derived sizes of a handle, passed by value to kernels.
struct Dims {
  int D, Hq, Hkv, dh, W, S, Hm, P, N, L, Bmax;
  int G;       // Hq / Hkv
  int QD;      // Hq*dh
  int KVD;     // Hkv*dh
  int dinner;  // Hm*P
  int Nd;      // draft projection columns: QD + 2*KVD + N
  int Nc;      // commit projection columns per layer: 2*KVD + dinner + N + Hm
  int NS;      // memory-input columns: dinner + N + Hm
  int Nz;      // output-projection inputs: QD + dinner
  int esize;   // element bytes of the model dtype
  int xoff;    // 1: cross-slot attention off (slot s sees the window and its own key)
  int Mh;      // memory horizon: 0 = whole history, M > 0 = last M committed features
  int Mr;      // rows of the memory-input ring (M > 1: M + S + 1, else 0)
  int gdn;     // 1: gated-delta memory (commit columns gain beta: Nc, NS + Hm)
  long long wait;  // limit (clock cycles) of the CUDA-core attention's ring-tile
                   // wait: kWaitCycles unless a test shortened it
  int blk;     // 1: full drafter block (norms, RoPE, conv, gate/skip, MLP, head)
  int F;       // block: MLP width
  int V;       // block: LM-head vocabulary
};

// ---------------------------------------------------------------- GEMM epilogues
enum EpiKind : int {
  EPI_F32 = 0,    // plain fp32 store
  EPI_RESID = 1,  // residual add, model dtype
  EPI_SSM_KV = 2, // ring append / memory inputs (commit, prefill window)
  EPI_DT = 3,     // prefill: dt of token r, head c, stored transposed (fp32)
  EPI_XB = 4,     // prefill: w-scaled x and B of token r, stored transposed (model dtype)
  EPI_STATE = 5,  // prefill: state row r = (head, p), column n: decay * state + v
  EPI_MEMRING = 6 // prefill, memory horizon M > 1: x / B / dt of the last M features
};

struct Epi {
  int kind;
  // EPI_F32: out[r*ld + c] = v
  float* out;
  int ld;
  // EPI_RESID: out_t[r*ld + c] = resid[r*ld + c] + v  (model dtype)
  const void* resid;
  void* out_t;
  // EPI_SSM_KV: column c -> layer = layer0 + c / cols_per_layer,
  // local column cl = c % cols_per_layer + col_off in the per-layer
  // [K | V | x | B | dt] block. K/V go to the ring slot of the row's
  // committed position; x, B and softplus(dt + bias) go to xbd (fp32).
  int layer0, cols_per_layer, col_off;
  int cols_valid;           // > 0: per-layer columns at or past this are padding (skipped)
  // Row source of EPI_SSM_KV (one of):
  //  * commit rows (n_acc != NULL): row r = b*(S+1) + t of the caller's
  //    [B, S+1, D] features; valid iff 0 <= n_acc[b] <= S+1 and t < n_acc[b];
  //    committed position pos[b] + t (pos before this commit);
  //  * mapped rows (row_req != NULL): request and position per packed row;
  //  * neither: every row valid, no ring columns (x/B/dt of prefill tokens).
  const int32_t* n_acc;
  const int64_t* pos;
  const int32_t* row_req;
  const int64_t* row_pos;
  void* ring_k;
  void* ring_v;
  float* xbd;
  long long xbd_layer_stride;  // elements between layers in xbd
  const float* dt_bias;        // [L][Hm]
  int64_t* pos_snap;           // commit rows: pos[b] before the commit, stored by row t = 0
  // EPI_MEMRING (mapped rows; columns [x | B | dt] of layer0): rows at
  // positions >= req_len[b] - Mh go to ring row (position mod Mr)
  float* mx;                   // [L][Bmax][Mr][dinner]
  float* mb;                   // [L][Bmax][Mr][N]
  float* mdt;                  // [L][Bmax][Hm][Mr]
  const int64_t* req_len;      // [Bmax]
  // Prefill chunked-scan epilogues (one request, one segment of T tokens):
  //  EPI_DT    dtw[c*ldt + r] = softplus(v + dt_bias[layer0][c])
  //  EPI_XB    c <  dinner: xsT[c*ldt + r] = dtw[(c/P)*ldt + r] * v   (dtw holds w)
  //            c >= dinner: bT[(c-dinner)*ldt + r] = v
  //  EPI_STATE st[r*N + c] = seg_decay[r/P] * st[r*N + c] + v
  float* dtw;
  int ldt;
  void* xsT;
  void* bT;
  float* st;
  const float* seg_decay;
  Dims d;
};

// Request and committed position of an EPI_SSM_KV row; position < 0: skip.
// c: the first output column the caller stores for this row (column 0 of a
// commit row t = 0 also records the position before the commit).
__device__ __forceinline__ void epi_row(const Epi& e, int r, int& b, long long& p, int c) {
  if (e.n_acc) {
    const int lim = e.d.S + 1;
    b = r / lim;
    const int t = r % lim;
    const int n = __ldcg(&e.n_acc[b]);
    p = (n >= 0 && n <= lim && t < n) ? __ldcg(&e.pos[b]) + t : -1;
    if (e.pos_snap && t == 0 && c == 0 && p >= 0) e.pos_snap[b] = p;
  } else if (e.row_req) {
    b = __ldcg(&e.row_req[r]);
    p = __ldcg(&e.row_pos[r]);
  } else {
    b = 0;
    p = 0;
  }
}

template <typename T>
__device__ __forceinline__ void epi_ssm(const Epi& e, int r, int c, float v, int b, long long p) {
  if (p < 0) return;
  const Dims& d = e.d;
  const int layer = e.layer0 + c / e.cols_per_layer;
  const int cl = c % e.cols_per_layer + e.col_off;
  if (e.cols_valid > 0 && cl >= e.cols_valid) return;
  if (cl < 2 * d.KVD) {
    const int which = cl >= d.KVD;
    const int cc = cl - which * d.KVD;
    const int kvh = cc / d.dh, dd = cc % d.dh;
    const int slot = (int)(p % d.W);
    const size_t idx = ((((size_t)layer * d.Bmax + b) * d.Hkv + kvh) * d.W + slot) * d.dh + dd;
    ((T*)(which ? e.ring_v : e.ring_k))[idx] = from_f<T>(v);
  } else {
    const int j = cl - 2 * d.KVD;
    float o = v;
    if (j >= d.dinner + d.N + d.Hm)
      o = sigmoid_f(v);
    else if (j >= d.dinner + d.N)
      o = softplus_f(v + __ldg(&e.dt_bias[layer * d.Hm + (j - d.dinner - d.N)]));
    e.xbd[(size_t)layer * e.xbd_layer_stride + (size_t)r * d.NS + j] = o;
  }
}

// The same epilogue split into a per-column part (fixed for a thread that
// owns one output column) and a per-row part (the ring-row offset of a
// committed row, -1 when the row is skipped), so that a tile's inner loop is
// one store per element.
struct SsmCol {
  int kind;      // 0: skip, 1: ring K/V, 2: x or B, 3: dt (softplus with bias), 4: beta (sigmoid)
  void* ring;    // ring_k or ring_v (kind 1)
  size_t base;   // element offset of (layer, head, dim) in the ring, or of (layer, column) in xbd
  float bias;    // dt bias (kind 3)
};

__device__ __forceinline__ SsmCol ssm_col(const Epi& e, int c) {
  const Dims& d = e.d;
  SsmCol k{0, nullptr, 0, 0.f};
  const int layer = e.layer0 + c / e.cols_per_layer;
  const int cl = c % e.cols_per_layer + e.col_off;
  if (e.cols_valid > 0 && cl >= e.cols_valid) return k;
  if (cl < 2 * d.KVD) {
    const int which = cl >= d.KVD;
    const int cc = cl - which * d.KVD;
    k.kind = 1;
    k.ring = which ? e.ring_v : e.ring_k;
    k.base = (((size_t)layer * d.Bmax * d.Hkv + cc / d.dh) * d.W) * d.dh + cc % d.dh;
  } else {
    const int j = cl - 2 * d.KVD;
    k.base = (size_t)layer * e.xbd_layer_stride + j;
    k.kind = 2;
    if (j >= d.dinner + d.N + d.Hm) {
      k.kind = 4;
    } else if (j >= d.dinner + d.N) {
      k.kind = 3;
      k.bias = __ldg(&e.dt_bias[layer * d.Hm + (j - d.dinner - d.N)]);
    }
  }
  return k;
}

// Ring-row offset of row r (request b, position p), or -1 when p < 0.
__device__ __forceinline__ long long ssm_row_off(const Dims& d, int b, long long p) {
  return p < 0 ? -1 : ((long long)b * d.Hkv * d.W + p % d.W) * d.dh;
}

template <typename T>
__device__ __forceinline__ void ssm_store(const Epi& e, const SsmCol& k, int r, long long ro,
                                          float v) {
  if (ro < 0 || k.kind == 0) return;
  if (k.kind == 1)
    static_cast<T*>(k.ring)[k.base + ro] = from_f<T>(v);
  else
    e.xbd[k.base + (size_t)r * e.d.NS] =
        k.kind == 3 ? softplus_f(v + k.bias) : (k.kind == 4 ? sigmoid_f(v) : v);
}

template <typename T>
__device__ __forceinline__ void epi_apply(const Epi& e, int r, int c, float v) {
  if (e.kind == EPI_F32) {
    e.out[(size_t)r * e.ld + c] = v;
  } else if (e.kind == EPI_RESID) {
    size_t i = (size_t)r * e.ld + c;
    float x = to_f(__ldcg(&((const T*)e.resid)[i]));
    ((T*)e.out_t)[i] = from_f<T>(x + v);
  } else if (e.kind == EPI_SSM_KV) {
    int b;
    long long p;
    epi_row(e, r, b, p, c);
    epi_ssm<T>(e, r, c, v, b, p);
  } else if (e.kind == EPI_DT) {
    e.dtw[(size_t)c * e.ldt + r] = softplus_f(v + __ldg(&e.dt_bias[e.layer0 * e.d.Hm + c]));
  } else if (e.kind == EPI_XB) {
    if (c < e.d.dinner) {
      const float w = __ldcg(&e.dtw[(size_t)(c / e.d.P) * e.ldt + r]);
      static_cast<T*>(e.xsT)[(size_t)c * e.ldt + r] = from_f<T>(w * v);
    } else {
      static_cast<T*>(e.bT)[(size_t)(c - e.d.dinner) * e.ldt + r] = from_f<T>(v);
    }
  } else if (e.kind == EPI_MEMRING) {
    const Dims& d = e.d;
    const int b = __ldcg(&e.row_req[r]);
    const long long p = __ldcg(&e.row_pos[r]);
    if (p < __ldcg(&e.req_len[b]) - d.Mh) return;  // older than the horizon
    const size_t lb = (size_t)e.layer0 * d.Bmax + b;
    const int row = (int)(p % d.Mr);
    if (c < d.dinner) {
      e.mx[(lb * d.Mr + row) * d.dinner + c] = v;
    } else if (c < d.dinner + d.N) {
      e.mb[(lb * d.Mr + row) * d.N + (c - d.dinner)] = v;
    } else if (c < d.dinner + d.N + d.Hm) {
      const int hd = c - d.dinner - d.N;
      e.mdt[(lb * d.Hm + hd) * d.Mr + row] =
          softplus_f(v + __ldg(&e.dt_bias[e.layer0 * d.Hm + hd]));
    }
  } else {  // EPI_STATE
    const size_t i = (size_t)r * e.d.N + c;
    e.st[i] = fmaf(__ldcg(&e.seg_decay[r / e.d.P]), __ldcg(&e.st[i]), v);
  }
}

// ------------------------------------------------- memory read, tensor cores
// y[s, p] = sum_n h[p, n] C[s, n] of one (request, memory head) as a
// [P x N] x [N x 8] product on mma.sync m16n8k8 tf32 (fp32 accumulate; h
// and C rounded to tf32 with round-to-nearest, relative error 2^-11, below
// the bf16 rounding of the output). Warp (m-tile, k-part) takes 16 state
// rows and N / parts columns; within each group of 16 columns lane t holds
// columns 4t..4t+3 and serves two k-steps (columns 4t, 4t+1 as logical
// k = t, t + 4, then 4t+2, 4t+3): the same permutation on both operands,
// so the sum is unchanged.
constexpr int MEM_G16 = 8;  // 16-column groups per warp (N <= 128)

__host__ __device__ inline bool mem_tc_ok(const Dims& d) {
  return d.P % 16 == 0 && d.P <= 128 && d.N % 16 == 0 && d.N <= 128 && d.S <= 8;
}
__host__ __device__ inline int mem_ksplit(const Dims& d) {
  const int mt = d.P / 16;
  int ks = mt >= 8 ? 1 : 8 / mt;
  while (ks > 1 && (d.N / 16) % ks) --ks;
  return ks;
}
// Sum over the 32 lanes of each of 32 values: after the butterfly each lane
// l holds the total of value l (31 shuffles instead of 32 x 5).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

// Staged heads per memory-read CTA of the attention launch (each as
// ceil(N / 32) swizzled 128-byte column groups of P rows), then the partial
// sums, 1/|C_s| (gated delta) and one barrier per buffer.
constexpr int MEM_NBUF = 3;
__host__ __device__ inline size_t mem_stage_bytes(const Dims& d) {
  return (size_t)((d.N + 31) / 32) * d.P * 128;
}
__host__ __device__ inline size_t mem_tc_bytes(const Dims& d) {
  return (size_t)MEM_NBUF * mem_stage_bytes(d) + (size_t)mem_ksplit(d) * d.P * 8 * 4 + 16 * 4 +
         MEM_NBUF * 8;
}

// Gated-delta read (q = C_s / |C_s|): 1/|C_s| of the S slot rows c0 + s*ld
// into qn[0..S), one warp per row; the caller synchronises before use.
__device__ __forceinline__ void slot_inv_norms(const float* c0, int ld, int S, int N, float* qn) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int s = warp; s < S; s += nw) {
    float acc = 0.f;
    for (int c = lane; c < N; c += 32) {
      const float v = __ldcg(&c0[(size_t)s * ld + c]);
      acc = fmaf(v, v, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) qn[s] = 1.f / sqrtf(acc);
  }
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_tf32_1688(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- launchers
// Every launcher enqueues on `st` and returns cudaGetLastError().

// Y[r, c] = sum_k X[r, k] * Wt[c, k] for r < R, c < C; epilogue per element.
// X row stride ldx, Wt row stride ldw (both in elements). part: split-K
// scratch of at least splits*R*C floats (unused when splits == 1).
cudaError_t launch_gemm_fma(int dtype, const void* X, int ldx, const void* Wt, int ldw,
                            int R, int C, int K, int splits, float* part,
                            const Epi& epi, cudaStream_t st, int* launches);

// bf16 tensor-core GEMM: D[m, n] = sum_k A[m, k] * B[n, k], A [M, K] with row
// stride lda, B [N, K] with row stride ldb (elements, multiples of 8). With
// swap = 1 the epilogue sees (row n, column m), else (row m, column n).
// Split-K partner CTAs (splits <= 8) form a thread-block cluster and sum
// their partial tiles through distributed shared memory.
// a_tiles (optional): A pre-tiled by tile_weights, read with bulk copies.
// late_trigger: the CTAs signal programmatic completion only after their own
// dependency wait, so that the next launch may read, before its own wait,
// anything that the launches before this one wrote.
// a_group_mtiles: a_tiles holds consecutive groups of that many m-tiles,
// each tiled on its own by tile_weights (one matrix per layer, stacked);
// 0: one matrix.
cudaError_t launch_gemm_tc(const void* A, long long lda, int M, const void* B, long long ldb,
                           int N, int K, int swap, int splits, int32_t* err, const Epi& epi,
                           cudaStream_t st, int* launches, const void* a_tiles = nullptr,
                           int late_trigger = 0, int a_group_mtiles = 0, int q4 = 0,
                           int independent = 0);
// Two swapped products with the same K in one launch (both A operands
// pre-tiled): D0 = A0 B0^T with epilogue epi0, D1 = A1 B1^T with epi1.
cudaError_t launch_gemm_tc_grouped(const void* a_tiles0, int M0, int gm0, const void* B0,
                                   long long ldb0, int N0, const Epi& epi0, const void* a_tiles1,
                                   int M1, const void* B1, long long ldb1, int N1, const Epi& epi1,
                                   int K, int splits, int32_t* err, cudaStream_t st, int* launches,
                                   int late_trigger = 0, int q4 = 0);

// 4-bit weights (GPTQ-style: codes 0..15, per row and 128-column group a bf16
// scale s and a zero point z, w = s * (code - z)), pre-tiled like
// tile_weights: per (m_tile, k_block) of 128 rows x 64 columns, 32 bytes of
// codes per row (one 32-bit word per 8 columns: nibble i holds column 2i for
// i < 4 and column 2(i-4)+1 otherwise), then per row one word (s's bf16 bits
// | z << 16). q4 launches read these tiles (skinny products, at most 32
// activation rows).
constexpr int Q4_TILE_BYTES = 128 * 32 + 128 * 4;
size_t q4_tiled_bytes(long long M, long long K);
// codes [M][K] (0..15), prm [M][K/128] (scale bits | zero << 16) -> tiles
void tile_weights_q4(const uint8_t* codes, const uint32_t* prm, long long M, long long K,
                     uint8_t* dst);
void tile_weights(const uint16_t* src, long long M, long long K, uint16_t* dst);

// Stream-K variant for the skinny swapped products (gemm_streamk.cu): one or
// two products with pre-tiled A (a_tiles1 = NULL: one), at most 32 activation
// rows each, the (m-tile, k-block) units split evenly over min(num_sms,
// units) CTAs; split tiles are summed through ws (floats) with one ticket
// per tile (tickets zero between launches, restored by every launch).
cudaError_t configure_gemm_sk();
// Workspace floats a launch of these shapes needs (tiles, slots per tile out).
size_t gemm_sk_workspace(int M0, int M1, int K, int num_sms, int* tiles, int* nslot);
// Token-major stream-K variant (gemm_streamk_tm.cu) for products with more
// than 32 activation rows: X [M, K] activation rows and W [N, K] plain
// weights through TMA, output row m (token), column n (feature); one or two
// products (X1 = NULL: one); ws: gemm_tm_workspace(num_sms) floats.
cudaError_t configure_gemm_tm();
size_t gemm_tm_workspace(int num_sms);
cudaError_t launch_gemm_tm(const void* X0, long long ldx0, int M0, const void* W0, long long ldw0,
                           int N0, const Epi& epi0, const void* X1, long long ldx1, int M1,
                           const void* W1, long long ldw1, int N1, const Epi& epi1, int K,
                           int num_sms, float* ws, size_t ws_floats, int* tickets, int n_tickets,
                           int32_t* err, int late_trigger, cudaStream_t st, int* launches);
cudaError_t launch_gemm_sk(const void* a_tiles0, int M0, int gm0, const void* B0, long long ldb0,
                           int N0, const Epi& epi0, const void* a_tiles1, int M1, const void* B1,
                           long long ldb1, int N1, const Epi& epi1, int K, int num_sms, float* ws,
                           size_t ws_floats, int* tickets, int n_tickets, int32_t* err,
                           int late_trigger, cudaStream_t st, int* launches);

// Persistent warp-specialised bf16 GEMM for large token-major products
// (gemm_persistent.cu): output row m of A's rows, column n of B's rows;
// epilogue through epi_chunk16. One CTA per SM (num_sms).
cudaError_t configure_tc_persistent(int num_sms);
cudaError_t launch_gemm_persistent(const void* A, long long lda, int M, const void* B,
                                   long long ldb, int N, int K, int32_t* err, const Epi& epi,
                                   int num_sms, cudaStream_t st, int* launches);
size_t tiled_bytes(long long M, long long K);
int tc_pick_splits(int M, int N, int K, int q4 = 0);

// 2-D bf16 tensor map over rows x K (row stride ld elements), box 64 x
// box_rows, 128-byte swizzle (gemm_tc.cu).
cudaError_t make_map(CUtensorMap* map, const void* base, long long rows, long long K, long long ld,
                     int box_rows);
// 2-D fp32 tensor map over rows x cols (row stride cols), box 32 columns x
// box_rows, 128-byte swizzle (gemm_tc.cu): the memory states of a layer,
// one box column group of a head per copy.
cudaError_t make_map_f32(CUtensorMap* map, const void* base, long long rows, long long cols,
                         int box_rows);

// One-time kernel attribute set-up (dynamic shared memory limits, driver
// entry points, cluster occupancy), done at handle creation.
cudaError_t configure_tc();
cudaError_t configure_attn_cluster(const Dims& d);

// Window+block attention and memory read for one layer, batch B, one launch
// (attention_cluster.cu). proj [B*S, Nd] fp32 (Q|K_s|V_s|C_s); ring_k/v and
// state of this layer; pos [Bmax]; mix [B*S, Nz] model dtype (O | y).
// bf16 handles with head_dim % 64 == 0 run the tensor-core variant, which
// loads ring tiles through the per-layer tensor maps mk / mv (rows =
// Bmax*Hkv*W, box attn_tile_rows(d) rows) and, when its memory read runs on
// the tensor cores (mem_tc_ok), the layer's states through ms (make_map_f32
// over rows Bmax*Hm*P, N columns, box P rows); other handles pass NULL maps.
// early: what the previous launch (which signalled its dependents after its
// own wait) leaves final at launch, read before this launch's wait:
// bit 0 the ring K/V, bit 1 the positions and states, bit 2 the slot
// projections (memory-read CTAs use bit 1 for state and C alike).
// with_mem = 0: attention only (the memory read was done elsewhere).
size_t attn_cluster_smem(const Dims& d, int esize);
int attn_tile_rows(const Dims& d);
bool attn_uses_tc(const Dims& d, int dtype);
cudaError_t launch_attn_cluster(int dtype, const Dims& d, int B, const float* proj,
                                const void* ring_k, const void* ring_v, const int64_t* pos,
                                const float* state, void* mix, const CUtensorMap* mk,
                                const CUtensorMap* mv, const CUtensorMap* ms, int32_t* err,
                                int num_sms, int early, int with_mem, cudaStream_t st,
                                int* launches);

// Commit state step, all layers: validates the accepted counts (error word),
// writes the packed offsets (exclusive scan of the valid counts) and the ring
// tags of the appended positions, advances the memory over rows
// b*(S+1) + t < b*(S+1) + n_b of xbd in order, then pos += n. memC (or
// NULL): C columns of the next draft's layer-0 slot projections (row
// stride Nd); the layer-0 memory read of that draft is then done here, on
// the new state, into the memory columns of mix (model dtype).
size_t commit_state_smem(const Dims& d, bool read);
cudaError_t configure_commit_state(const Dims& d);  // at handle creation
// Memory-input ring of a memory horizon M > 1 (all NULL otherwise): x / B /
// dt of the last Mr = M + S + 1 committed features per (layer, request),
// position t in row t mod Mr, and the positions before the running commit
// (stored by the commit projection's epilogue).
struct MemRing {
  float* x;          // [L][Bmax][Mr][dinner]
  float* b;          // [L][Bmax][Mr][N]
  float* dt;         // [L][Bmax][Hm][Mr]
  const int64_t* pos_snap;  // [Bmax]
};

cudaError_t launch_commit_state(int dtype, const Dims& d, int B, const int32_t* n_acc,
                                const float* xbd, long long xbd_layer_stride, const float* A_log,
                                float* state, int64_t* pos, int32_t* offsets, int32_t* tags,
                                int32_t* err, const float* memC, void* mix, int early,
                                int late, int num_sms, const MemRing& mr, cudaStream_t st);

// Prefill helpers (lens/reqs/cu are device int32 arrays of n_req entries).
cudaError_t launch_prefill_reset(const Dims& d, int n_req, const int32_t* reqs,
                                 float* state, int32_t* tags, int64_t* pos, cudaStream_t st);
// Gated-delta prefill of request b, layer `layer`: the T rows of xs (x | B |
// dt | beta, stride NS, as the commit projection writes them) applied in
// order to the state.
cudaError_t launch_gdn_prefill(const Dims& d, int layer, int b, int T, const float* xs,
                               const float* A_log, float* state, cudaStream_t st);

// (req_len, when not NULL, receives each named request's prefix length.)
cudaError_t launch_prefill_ring_prep(int dtype, const Dims& d, int n_req, int n_rows,
                                     const int32_t* lens, const int32_t* reqs,
                                     const void* feats, int32_t* row_req, int64_t* row_pos,
                                     int32_t* tags, void* packed, int64_t* req_len,
                                     cudaStream_t st);
// Chunked decay scan of one prefill segment of T tokens, per head h (grid Hm):
// dtw[h][t] holds dt_t on entry and w_t = dt_t * exp(A_h * sum_{s>t} dt_s)
// on exit; seg_decay[h] = exp(A_h * sum_t dt_t). Chunks of `chunk` tokens
// are scanned within a warp; chunk and warp totals combine with shuffles
// and a CTA-level suffix pass.
cudaError_t launch_prefill_decay(const Dims& d, int layer, int T, int ldt, int chunk, float* dtw,
                                 const float* A_log, float* seg_decay, cudaStream_t st);
// Message reported by hf_last_error(NULL) for calls that have no handle.
void set_thread_error(const char* msg);

// full drafter block (block.cu)
cudaError_t launch_rms_norm(int dtype, const void* x, const float* g, void* y, int rows, int D,
                            cudaStream_t st);
cudaError_t launch_rope_slots(const Dims& d, int rows, float* proj, const int64_t* pos,
                              const double* inv, cudaStream_t st);
cudaError_t launch_gate_skip(int dtype, const Dims& d, int rows, void* mix, const float* proj,
                             const float* d_skip, cudaStream_t st);
cudaError_t launch_swiglu(int dtype, int rows, int F, const float* h, void* act, cudaStream_t st);
cudaError_t launch_argmax(int rows, int V, const float* logits, int32_t* tokens, cudaStream_t st);
cudaError_t launch_commit_prep(int dtype, const Dims& d, int B, const int32_t* n_acc,
                               const int64_t* pos, void* ring_k, float* xbd, long long xls,
                               float* conv_state, const float* conv_w, const float* conv_b,
                               const double* inv, cudaStream_t st);
cudaError_t launch_ring_rope(int dtype, const Dims& d, int layer, int rows, const int32_t* row_req,
                             const int64_t* row_pos, void* ring_k, const double* inv,
                             cudaStream_t st);
cudaError_t launch_conv_prefill(int dtype, const Dims& d, int Tn, int ldt, const float* U,
                                float* hist, const float* dtw, const float* conv_w,
                                const float* conv_b, void* xsT, void* bT, cudaStream_t st);
cudaError_t launch_conv_reset(const Dims& d, int n_req, const int32_t* reqs, float* conv_state,
                              cudaStream_t st);
// limit of hf_attention_noalloc's ring-tile waits (clock cycles; 0 = give up
// at once, the failure-detection tests' hook)
void set_noalloc_wait_limit(long long cycles);

cudaError_t launch_prefill_finish(int n_req, const int32_t* lens, const int32_t* reqs,
                                  int64_t* pos, cudaStream_t st);

}  // namespace hf
