// bf16 GEMM on the 5th-generation tensor cores: D[m, n] = sum_k A[m, k] * B[n, k].
//
// A and B are K-major bf16 matrices in global memory. TMA copies 64-wide
// K slices of both into 128-byte-swizzled shared memory (a ring of STAGES
// slots guarded by mbarriers), one elected thread issues tcgen05.mma
// (M = 128, N = BN, K = 16 per instruction) into an fp32 accumulator in
// tensor memory, and all four warps read the accumulator back with
// tcgen05.ld for the epilogue.
//
// Two uses:
//  * skinny (draft / commit): A = weights [out features, K], B = the few
//    activation rows (7 slots per request, or the accepted rows), so the
//    weights stream through the tensor core exactly once; the epilogue maps
//    D[m, n] to output row n, column m ("swap").
//  * token-major (more than 32 activation rows, prefill): A = the rows
//    [tokens, K], B = weight rows; output row m, column n.
// Split-K partners of one output tile form a thread-block cluster (along
// grid x) and sum their partial tiles through distributed shared memory in
// rank order (deterministic, no atomics on data): swap tiles by remote
// reads of the partners' partials, token-major tiles by pushing each
// partial chunk to the rank that owns it (remote stores, one exchange).
//
// Every mbarrier wait is bounded (clock-based); on expiry the CTA raises
// ERR_TIMEOUT in the device error word, drains the copies it issued (again
// bounded), frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace hf {
namespace {

// Thread-block-cluster helpers (split-K partner CTAs of one output tile form
// a cluster along grid z; partial tiles are summed through distributed
// shared memory).
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
__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Remote shared-memory store of four floats into partner `rank`'s copy of
// the local address (a cluster-window address; no reply is awaited).
__device__ __forceinline__ void st_peer4(const float* local, uint32_t rank, float4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// Receive slots of the token-major split-K sum: for (sending partner's slot,
// owned chunk k, tile row m) the row's 16 partial sums, its four float4 in
// an order rotated by row pair (conflict-free stores and loads by a warp of
// 32 consecutive rows). Returns the float offset of float4 q.
__device__ __forceinline__ int recv_off(int slot, int k, int kmax, int m, int q) {
  return (((slot * kmax + k) * 128 + m) << 4) + ((q ^ ((m >> 1) & 3)) << 2);
}

struct TcArgs {
  int M, N, K;        // D is M x N
  int kblocks;        // ceil(K / 64)
  int splits;         // split-K factor (grid.x = cluster size along x; <= 8)
  int swap;           // 1: output row = n, column = m; 0: row = m, column = n
  int prefetch_a;     // 1: A does not depend on earlier kernels (weights): load it
                      //    before waiting on the previous kernel
  const uint8_t* a_tiles;  // non-NULL: A stored pre-tiled (see tile_weights); each
                           // (m_tile, k_block) is one 16 KB swizzled tile, read by
                           // one bulk copy; NULL: A read through the tensor map
  int32_t* err;       // device error word
  int late_trigger;   // 1: signal dependents only after the dependency wait
  int independent;    // 1: neither operand depends on earlier kernels (both are inputs
                      //    of the call): the main loop runs without the dependency
                      //    wait; only the epilogue waits
  // Grouped launch: m-tiles [mt0, ...) belong to a second product with the
  // same K (its own A tiles, B map, N and epilogue). mt0 = all m-tiles when
  // there is one product.
  int mt0;
  int M1, N1;
  const uint8_t* a_tiles1;
  // Tiled A stored as consecutive groups of this many m-tiles (one matrix
  // tiled per layer, stacked), each group [k_block][m_tile]; per product.
  int a_gm0, a_gm1;
};

// Epilogue cache (shared memory after the barriers): per output row of the
// tile its request and committed position (ring rows), and for small tiles
// the residual inputs; filled during the main loop by the otherwise idle
// warps 2-3, so the epilogue issues no dependent global loads.
template <int BN>
struct EpiCache {
  static constexpr int RES_ROWS = BN <= 32 ? BN : 0;
  static constexpr size_t bytes = BN * 8 + BN * 4 + RES_ROWS * 128 * 4;
};

__device__ __forceinline__ __nv_bfloat162 bf2_of(uint32_t u) {
  __nv_bfloat162 v;
  memcpy(&v, &u, 4);
  return v;
}
__device__ __forceinline__ uint32_t bits_of(__nv_bfloat162 v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  return u;
}

// Q4: A is 4-bit weights (pre-tiled, Q4_TILE_BYTES per (m_tile, k_block):
// codes of 128 rows x 64 columns, then per row the bf16 scale and the zero
// point of its 128-column group). Warps 4-11 turn each packed tile into the
// bf16 swizzled tile the tensor core reads (w = scale * (code - zero), one
// rounding) and release it to the MMA warp through afull; the producer, MMA
// and epilogue warps are those of the bf16 kernel.
template <int BN, int STAGES, bool Q4>
__global__ void __launch_bounds__(Q4 ? 384 : 128, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb0,
               const __grid_constant__ CUtensorMap tb1, TcArgs a, const __grid_constant__ Epi epi0,
               const __grid_constant__ Epi epi1) {
  constexpr int A_BYTES = 128 * 128;
  constexpr int B_BYTES = BN * 128;
  constexpr int PK_BYTES = Q4 ? Q4_TILE_BYTES : 0;
  constexpr int TILE_BYTES = Q4 ? Q4_TILE_BYTES : A_BYTES;  // one stored A tile
  constexpr uint32_t STAGE_BYTES = TILE_BYTES + B_BYTES;    // bytes the copies of a stage bring
  constexpr uint32_t NCOLS = BN < 32 ? 32 : BN;
  constexpr int RES_ROWS = EpiCache<BN>::RES_ROWS;
  // Split-K partial tiles are summed through the drained stage buffers, 128
  // floats per tile column (token-major) or row (swap); when BN of them do
  // not fit (two-stage rings) the sum runs in passes of RED_COLS.
  constexpr int RED_FLOATS = STAGES * (A_BYTES + B_BYTES + PK_BYTES) / 4;
  constexpr int RED_COLS = (RED_FLOATS / 128 / 16) * 16 < BN ? (RED_FLOATS / 128 / 16) * 16 : BN;
  constexpr int RED_PASSES = (BN + RED_COLS - 1) / RED_COLS;
  static_assert(RED_COLS >= 16, "stage buffers too small for the split-K sum");
  // token-major split-K: (splits - 1) receive slots of ceil(chunks / splits)
  // 16-column chunks x 128 rows, for every cluster size up to 8
  constexpr int NCH = BN / 16 > 0 ? BN / 16 : 1;
  static_assert(7 * ((NCH + 6) / 7) * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES) &&
                    6 * ((NCH + 5) / 6) * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES) &&
                    5 * ((NCH + 4) / 5) * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES) &&
                    4 * ((NCH + 3) / 4) * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES) &&
                    3 * ((NCH + 2) / 3) * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES) &&
                    2 * ((NCH + 1) / 2) * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES) &&
                    NCH * 8192 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES),
                "stage buffers too small for the split-K receive slots");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sP = sB + STAGES * B_BYTES;  // Q4: packed tiles
  uint64_t* full = reinterpret_cast<uint64_t*>(sP + STAGES * PK_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* afull = empty + STAGES;     // Q4: dequantised A tile ready
  uint64_t* done = afull + (Q4 ? STAGES : 0);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] issued, [2] consumed, [3] last
  // epilogue cache after the 32 bytes of TMEM slot and flags (8-byte aligned)
  long long* ep_p = reinterpret_cast<long long*>(reinterpret_cast<uint8_t*>(done) + 8 + 32);
  int* ep_b = reinterpret_cast<int*>(ep_p + BN);
  float* ep_res = reinterpret_cast<float*>(ep_b + BN);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // grid (splits, m_tiles, n_tiles); the splits of one tile form a cluster along x
  const int split = blockIdx.x, n_tile = blockIdx.z;
  const bool second = (int)blockIdx.y >= a.mt0;  // tile of the second product
  const int m_tile = second ? (int)blockIdx.y - a.mt0 : (int)blockIdx.y;
  const int M = second ? a.M1 : a.M, N = second ? a.N1 : a.N;
  const uint8_t* a_tiles = second ? a.a_tiles1 : a.a_tiles;
  const int a_gm = second ? a.a_gm1 : a.a_gm0;  // m-tiles per stored group
  const size_t a_tile_idx0 = ((size_t)(m_tile / a_gm) * a.kblocks) * a_gm + m_tile % a_gm;
  const bool epw = !Q4 || warp < 4;  // the warps of the epilogue (TMEM lane quadrants)
  const CUtensorMap* tb = second ? &tb1 : &tb0;
  const Epi& epi = second ? epi1 : epi0;
  if (n_tile * BN >= N) return;  // the other product has more n-tiles (whole cluster)
  const int kb0 = (int)((long long)split * a.kblocks / a.splits);
  const int kb1 = (int)((long long)(split + 1) * a.kblocks / a.splits);
  const int nkb = kb1 - kb0;
  if (!a.late_trigger) pdl_trigger();

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if (Q4) mbar_init(&afull[s], 8);  // one arrival per dequantising warp
    }
    mbar_init(done, 1);
    flags[0] = flags[1] = flags[2] = flags[3] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(NCOLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer. The first ring of stages is filled up front; with
    // prefetch_a the A tiles (weights) are requested before waiting for the
    // previous kernel, so their HBM read overlaps that kernel's tail.
    const int pre = nkb < STAGES ? nkb : STAGES;
    // A tile of local k-block i into stage st
    auto load_a = [&](int st, int i) {
      if (Q4)
        bulk_g2s(sP + st * PK_BYTES,
                 a_tiles + (a_tile_idx0 + (size_t)(kb0 + i) * a_gm) * (size_t)TILE_BYTES,
                 TILE_BYTES, &full[st]);
      else if (a_tiles)
        bulk_g2s(sA + st * A_BYTES,
                 a_tiles + (a_tile_idx0 + (size_t)(kb0 + i) * a_gm) * (size_t)A_BYTES, A_BYTES,
                 &full[st]);
      else
        tma_load_2d(sA + st * A_BYTES, &ta, &full[st], (kb0 + i) * 64, m_tile * 128);
    };
    if (a.independent) {
      for (int j = 0; j < pre; ++j) {
        mbar_expect_tx(&full[j], STAGE_BYTES);
        load_a(j, j);
        tma_load_2d(sB + j * B_BYTES, tb, &full[j], (kb0 + j) * 64, n_tile * BN);
      }
    } else if (a.prefetch_a) {
      for (int j = 0; j < pre; ++j) {
        mbar_expect_tx(&full[j], STAGE_BYTES);
        load_a(j, j);
      }
      pdl_wait();
      if (a.late_trigger) pdl_trigger();
      for (int j = 0; j < pre; ++j)
        tma_load_2d(sB + j * B_BYTES, tb, &full[j], (kb0 + j) * 64, n_tile * BN);
    } else {
      pdl_wait();
      if (a.late_trigger) pdl_trigger();
      for (int j = 0; j < pre; ++j) {
        mbar_expect_tx(&full[j], STAGE_BYTES);
        load_a(j, j);
        tma_load_2d(sB + j * B_BYTES, tb, &full[j], (kb0 + j) * 64, n_tile * BN);
      }
    }
    int i = pre;
    for (; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (i >= STAGES && !mbar_wait(&empty[s], ph ^ 1u)) {
        atomicExch(&flags[0], 1);
        break;
      }
      if (*(volatile int*)&flags[0]) break;
      mbar_expect_tx(&full[s], STAGE_BYTES);
      load_a(s, i);
      tma_load_2d(sB + s * B_BYTES, tb, &full[s], (kb0 + i) * 64, n_tile * BN);
    }
    flags[1] = i;
  } else if (a.late_trigger && !a.independent) {
    pdl_wait();
    pdl_trigger();
  }
  if (Q4 && warp >= 4) {
    // dequantisers: thread (r, h) makes columns 32h..32h+31 of tile row r
    const int dq = tid - 128, r = dq >> 1, h = dq & 1;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      if (!mbar_wait(&full[s], (uint32_t)(i / STAGES) & 1u)) {
        atomicExch(&flags[0], 1);
        break;
      }
      const uint8_t* pk = sP + s * PK_BYTES;
      const uint4 cw = *reinterpret_cast<const uint4*>(pk + r * 32 + h * 16);
      const uint32_t prm = *reinterpret_cast<const uint32_t*>(pk + 4096 + r * 4);
      // bf16 pairs: s in both halves; 128 + z in both halves (0x4300 | z)
      const uint32_t sb = prm & 0xFFFFu, zb = 0x4300u | ((prm >> 16) & 0xFu);
      const __nv_bfloat162 s2 = bf2_of(sb | (sb << 16)), c2 = bf2_of(zb | (zb << 16));
      const uint32_t wds[4] = {cw.x, cw.y, cw.z, cw.w};
      uint8_t* arow = sA + s * A_BYTES + r * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int c = 4 * h + cc;  // 16-byte chunk: columns 8c..8c+7
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // nibbles j and j + 4 of the word are columns 8c + 2j and 8c + 2j + 1
          // (the tiles store them so); OR-ing a nibble into 0x4300 makes the
          // bf16 128 + code, minus 128 + z is code - z exactly, times s rounds once
          const uint32_t x = ((wds[cc] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
          o[j] = bits_of(__hmul2(__hsub2(bf2_of(x), c2), s2));
        }
        *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for the tensor core
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&afull[s])) : "memory");
    }
  }
  if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16(BN < 16 ? 16 : BN);
    uint64_t* ready = Q4 ? afull : full;
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait(&ready[s], ph)) {
        atomicExch(&flags[0], 1);
        break;
      }
      tc_fence_after();
      const uint64_t da = sdesc_sw128(sA + s * A_BYTES);
      const uint64_t db = sdesc_sw128(sB + s * B_BYTES);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem, da + 2ull * kk, db + 2ull * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&empty[s]);
    }
    flags[2] = i;
    umma_commit(done);
  }
  __syncwarp();
  pdl_wait();  // the epilogue writes memory earlier kernels may still read
  if (a.independent && a.late_trigger) pdl_trigger();
  const int n_here = min(BN, N - n_tile * BN);
  if (warp >= 2 && epw && a.swap) {  // idle during the main loop: fetch the epilogue inputs
    const int t2 = tid - 64;
    if (epi.kind == EPI_SSM_KV) {
      for (int nl = t2; nl < n_here; nl += 64) {
        int bq;
        long long pq;
        epi_row(epi, n_tile * BN + nl, bq, pq, m_tile * 128);
        ep_b[nl] = bq;
        ep_p[nl] = ssm_row_off(epi.d, bq, pq);
      }
    } else if (epi.kind == EPI_RESID && RES_ROWS > 0) {
      const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(epi.resid);
      for (int i = t2; i < n_here * 128; i += 64) {
        const int nl = i >> 7, mq = m_tile * 128 + (i & 127);
        ep_res[i] = mq < M ? to_f(__ldcg(&res[(size_t)(n_tile * BN + nl) * epi.ld + mq])) : 0.f;
      }
    }
  }

  // token-major commit epilogue: the row's ring offset once per row (its
  // dependent loads overlap the main loop)
  const bool kv_tm = !a.swap && epi.kind == EPI_SSM_KV;
  const int m_row = m_tile * 128 + warp * 32 + lane;
  const long long ro_tm = kv_tm && epw && m_row < M ? ssm_kv_row(epi, m_row, n_tile * BN) : -1;

  const bool ok = mbar_wait(done, 0);
  if (__syncthreads_or(!ok || flags[0])) {
    // Timed out somewhere: report, drain issued copies (bounded), free TMEM.
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      for (int i = flags[2]; i < flags[1]; ++i)
        mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (a.splits > 1)  // keep the cluster's barrier sequence matched (token-major:
                       // two; swap: two per pass)
      for (int p = 0; p < (a.swap ? RED_PASSES : 1); ++p) {
        cluster_sync_all();
        cluster_sync_all();
      }
    if (warp == 1)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOLS));
    return;
  }
  tc_fence_after();

  const int m_local = warp * 32 + lane;
  const int m = m_tile * 128 + m_local;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  float v[16];
  // this thread's output column of the commit projection (swap only)
  const SsmCol scol = (a.swap && epi.kind == EPI_SSM_KV && m < M) ? ssm_col(epi, m)
                                                                      : SsmCol{0, nullptr, 0, 0.f};
  // Output of tile row nl (activation row n) and this thread's column m.
  auto emit = [&](int nl, float val) {
    const int n = n_tile * BN + nl;
    if (!a.swap) {
      epi_apply<__nv_bfloat16>(epi, m, n, val);
    } else if (epi.kind == EPI_F32) {
      epi.out[(size_t)n * epi.ld + m] = val;
    } else if (epi.kind == EPI_RESID) {
      const size_t i = (size_t)n * epi.ld + m;
      const float x = RES_ROWS > 0 ? ep_res[nl * 128 + m_local]
                                   : to_f(__ldcg(&static_cast<const __nv_bfloat16*>(epi.resid)[i]));
      static_cast<__nv_bfloat16*>(epi.out_t)[i] = __float2bfloat16_rn(x + val);
    } else if (epi.kind == EPI_SSM_KV) {
      ssm_store<__nv_bfloat16>(epi, scol, n, ep_p[nl], val);
    } else {  // any other epilogue: element (row n, column m)
      epi_apply<__nv_bfloat16>(epi, n, m, val);
    }
  };
  // token-major fp32 output: each warp stages its 32 rows in the drained
  // stage buffers and stores them a row at a time (the warp's 16-byte pieces
  // contiguous) instead of 32 rows' pieces per store instruction
  constexpr int FRS = BN + 4;  // staged row stride (floats): conflict-free
  static_assert(4 * 32 * FRS * 4 <= STAGES * (A_BYTES + B_BYTES + PK_BYTES),
                "stage buffers too small for the staged fp32 epilogue");
  const bool f32_rows = !a.swap && epi.kind == EPI_F32 && epi.ld % 4 == 0 && n_here % 4 == 0;
  if (a.splits == 1 && f32_rows) {
    if (epw) {
      float* stg = reinterpret_cast<float*>(smem) + (size_t)warp * 32 * FRS;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        tmem_ld16(trow + c0, v);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(&stg[lane * FRS + c0 + 4 * q]) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      __syncwarp();
      const int nv = n_here / 4;
#pragma unroll 1
      for (int r = 0; r < 32; ++r) {
        const int mr = m_tile * 128 + warp * 32 + r;
        if (mr >= M) break;
        float4* o = reinterpret_cast<float4*>(epi.out + (size_t)mr * epi.ld + n_tile * BN);
        for (int q = lane; q < nv; q += 32) o[q] = *reinterpret_cast<const float4*>(&stg[r * FRS + 4 * q]);
      }
    }
  } else if (a.splits == 1) {
#pragma unroll 1
    for (int c0 = 0; c0 < (epw ? BN : 0); c0 += 16) {
      tmem_ld16(trow + c0, v);
      if (m < M && c0 < n_here) {
        if (kv_tm) {
          epi_ssm_chunk16(epi, m, n_tile * BN + c0, min(16, n_here - c0), v, ro_tm);
        } else if (!a.swap) {
          epi_chunk16(epi, m, n_tile * BN + c0, min(16, n_here - c0), v);
        } else if (epi.kind == EPI_RESID && RES_ROWS == 0) {
          // 16 independent residual loads in flight, then the stores
          const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(epi.resid);
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(epi.out_t);
          const size_t base = (size_t)(n_tile * BN + c0) * epi.ld + m;
          float x[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            x[j] = c0 + j < n_here ? to_f(__ldcg(&res[base + (size_t)j * epi.ld])) : 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < n_here) out[base + (size_t)j * epi.ld] = __float2bfloat16_rn(x[j] + v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < n_here) emit(c0 + j, v[j]);
        }
      }
    }
  } else if (!a.swap) {
    // Split-K, token-major: 16-column chunk u of the tile belongs to rank
    // u % splits. Once every partner's main loop has drained (first cluster
    // barrier: the stage buffers are free), each partner pushes its partial
    // of the chunks it does not own into the owner's receive slots with
    // remote stores; after the second barrier the owner adds the partials in
    // rank order (its own straight from tensor memory; deterministic) and
    // runs the epilogue. The residual rows of the owned chunks are loaded
    // while the pushes are in flight.
    float* recv = reinterpret_cast<float*>(smem);
    const int rank = (int)cluster_rank(), S = a.splits;
    const int nch = (n_here + 15) / 16, kmax = (NCH + S - 1) / S;
    const bool resid = epi.kind == EPI_RESID && epi.ld % 8 == 0;
    constexpr int KPRE = (NCH + 1) / 2;  // owned chunks per rank, at most (S >= 2)
    uint4 rpre[2 * KPRE];
    if (epw && resid && m < M) {
#pragma unroll
      for (int k = 0; k < KPRE; ++k) {
        const int u = rank + k * S;
        if (u < nch && u * 16 + 16 <= n_here) {
          const uint4* r = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(epi.resid) + (size_t)m * epi.ld + n_tile * BN + u * 16);
          rpre[2 * k] = __ldcg(r);
          rpre[2 * k + 1] = __ldcg(r + 1);
        }
      }
    }
    cluster_sync_all();
    if (epw) {
#pragma unroll 1
      for (int u = 0; u < nch; ++u) {
        const int owner = u % S;
        if (owner == rank) continue;
        tmem_ld16(trow + u * 16, v);
        if (m < M) {
          const int slot = rank < owner ? rank : rank - 1, k = u / S;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_peer4(recv + recv_off(slot, k, kmax, m_local, q), (uint32_t)owner,
                     make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
        }
      }
    }
    cluster_sync_all();  // the pushed partials are visible to their owners
    if (epw) {
#pragma unroll 1
      for (int k = 0; k < kmax; ++k) {
        const int u = rank + k * S;
        if (u >= nch) break;
        float own[16];
        tmem_ld16(trow + u * 16, own);
        if (m < M) {  // a structured branch: the warp reconverges before the next tcgen05.ld
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.f;
          for (int sp = 0; sp < S; ++sp) {
            if (sp == rank) {
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] += own[j];
            } else {
              const int slot = sp < rank ? sp : sp - 1;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 p = *reinterpret_cast<const float4*>(recv + recv_off(slot, k, kmax, m_local, q));
                v[4 * q] += p.x;
                v[4 * q + 1] += p.y;
                v[4 * q + 2] += p.z;
                v[4 * q + 3] += p.w;
              }
            }
          }
          const int n0 = n_tile * BN + u * 16, nc = min(16, n_here - u * 16);
          bool pre = false;
#pragma unroll
          for (int kk = 0; kk < KPRE; ++kk)
            if (kk == k && resid && nc == 16) {
              epi_resid16(epi, m, n0, v, rpre[2 * kk], rpre[2 * kk + 1]);
              pre = true;
            }
          if (kv_tm)
            epi_ssm_chunk16(epi, m, n0, nc, v, ro_tm);
          else if (!pre)
            epi_chunk16(epi, m, n0, nc, v);
        }
      }
    }
  } else {
    // Split-K: this CTA's partial tile goes to its own shared memory (the
    // drained stage buffers); after a cluster barrier, rank r sums rows
    // r, r + splits, ... over all partners in rank order (deterministic).
    float* red = reinterpret_cast<float*>(smem);
    const int rank = (int)cluster_rank();
#pragma unroll 1
    for (int p0 = 0; p0 < BN; p0 += RED_COLS) {  // tile rows [p0, p0 + RED_COLS) per pass
      const int p1 = p0 + RED_COLS < BN ? p0 + RED_COLS : BN;
#pragma unroll 1
      for (int c0 = p0; c0 < (epw ? p1 : p0); c0 += 16) {
        tmem_ld16(trow + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < n_here) red[(c0 - p0 + j) * 128 + m_local] = v[j];
      }
      cluster_sync_all();
      const int pe = p1 < n_here ? p1 : n_here;
      for (int nl = p0 + rank; nl < (epw ? pe : p0); nl += a.splits) {
        float part[8];
#pragma unroll
        for (int sp = 0; sp < 8; ++sp)
          part[sp] = sp < a.splits ? ld_peer(&red[(nl - p0) * 128 + m_local], (uint32_t)sp) : 0.f;
        float sum = 0.f;
#pragma unroll
        for (int sp = 0; sp < 8; ++sp) sum += part[sp];
        if (m < M) emit(nl, sum);
      }
      cluster_sync_all();  // partners keep their shared memory until all reads are done
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOLS));
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      g_encode_err = e != cudaSuccess ? e : cudaErrorNotSupported;
    else
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode_err;
}

}  // namespace

// 2-D bf16 tensor map over rows x K (row stride ld elements), box 64 x box_rows,
// 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, const void* base, long long rows, long long K, long long ld,
                     int box_rows) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D fp32 tensor map over rows x cols (row stride cols elements, a multiple
// of 4), box 32 columns (128 bytes) x box_rows, 128-byte swizzle.
cudaError_t make_map_f32(CUtensorMap* map, const void* base, long long rows, long long cols,
                         int box_rows) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * 4)};
  cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// Pipeline depth of the narrow tiles (skinny products at small batch): a
// deep ring (one CTA per SM, ~130 KB in flight); 5 / 4 stages (two CTAs per
// SM) measured slower at batch 1.
constexpr int kStages16 = 7, kStages32 = 6;

template <int BN, int STAGES, bool Q4 = false>
constexpr size_t tc_smem() {
  // 1 KB alignment slack, stages (+ packed tiles), barriers, TMEM slot + flags
  // (28 B), epilogue cache
  return 1024 + (size_t)STAGES * (128 * 128 + BN * 128 + (Q4 ? Q4_TILE_BYTES : 0)) +
         ((Q4 ? 3 : 2) * STAGES + 1) * 8 + 32 + EpiCache<BN>::bytes;
}

template <int BN, int STAGES, bool Q4 = false>
cudaError_t configure_one() {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, Q4>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc_smem<BN, STAGES, Q4>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, Q4>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

template <int BN, int STAGES, bool Q4 = false>
cudaLaunchConfig_t tc_config(dim3 grid, int cz, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Q4 ? 384 : 128);
  cfg.dynamicSmemBytes = tc_smem<BN, STAGES, Q4>();
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cz;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int BN, int STAGES, bool Q4 = false>
cudaError_t launch_tc(const CUtensorMap& ma, const CUtensorMap& mb0, const CUtensorMap& mb1,
                      const TcArgs& a, const Epi& epi0, const Epi& epi1, dim3 grid,
                      cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = tc_config<BN, STAGES, Q4>(grid, a.splits, st, attr);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, STAGES, Q4>, ma, mb0, mb1, a, epi0, epi1);
}

// 4-bit weights: the skinny widths only (16 or 32 activation rows), the
// bf16 ring depths (one CTA per SM). A 4-stage ring with two CTAs per SM and
// split-K partners measured faster on the Phi-4 round projection (55 vs
// 74 us) but slower over the Qwen3-4B round (17.6K vs 18.9K steps/s).
template <typename... X>
cudaError_t launch_bn_q4(int bn, X&&... x) {
  switch (bn) {
    case 16: return launch_tc<16, kStages16, true>(x...);
    case 32: return launch_tc<32, kStages32, true>(x...);
  }
  return cudaErrorInvalidValue;
}

template <typename... X>
cudaError_t launch_bn(int bn, X&&... x) {
  switch (bn) {
    case 16: return launch_tc<16, kStages16>(x...);
    case 32: return launch_tc<32, kStages32>(x...);
    case 64: return launch_tc<64, 5>(x...);
    case 128: return launch_tc<128, 4>(x...);
    default: return launch_tc<256, 4>(x...);
  }
}

// How many clusters of cz CTAs of this instantiation are resident at once
// (the driver's answer for the tcgen05 kernel itself: one CTA per SM).
template <int BN, int STAGES, bool Q4 = false>
int max_clusters(int cz) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = tc_config<BN, STAGES, Q4>(dim3(cz, 1, 1), cz, nullptr, attr);
  cfg.attrs = attr + 1;  // occupancy query: cluster shape only
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<BN, STAGES, Q4>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int g_max_clusters[5][9] = {};  // [log2(BN/16)][cz]
int g_max_clusters_q4[2][9] = {};  // 4-bit variants, BN 16 and 32

}  // namespace

// Shared-memory limits of every instantiation, set at handle creation so
// that launches stay legal inside stream capture.
cudaError_t configure_tc() {
  cudaError_t e = get_encoder();
  if (e == cudaSuccess) e = configure_one<16, kStages16>();
  if (e == cudaSuccess) e = configure_one<32, kStages32>();
  if (e == cudaSuccess) e = configure_one<64, 5>();
  if (e == cudaSuccess) e = configure_one<128, 4>();
  if (e == cudaSuccess) e = configure_one<256, 4>();
  if (e == cudaSuccess) e = configure_one<16, kStages16, true>();
  if (e == cudaSuccess) e = configure_one<32, kStages32, true>();
  if (e != cudaSuccess) return e;
  for (int cz = 1; cz <= 8; ++cz) {
    g_max_clusters[0][cz] = max_clusters<16, kStages16>(cz);
    g_max_clusters[1][cz] = max_clusters<32, kStages32>(cz);
    g_max_clusters[2][cz] = max_clusters<64, 5>(cz);
    g_max_clusters[3][cz] = max_clusters<128, 4>(cz);
    g_max_clusters[4][cz] = max_clusters<256, 4>(cz);
    g_max_clusters_q4[0][cz] = max_clusters<16, kStages16, true>(cz);
    g_max_clusters_q4[1][cz] = max_clusters<32, kStages32, true>(cz);
  }
  return cudaSuccess;
}

// Split-K factor for an M x N x K product: the largest cluster size (<= 8,
// <= kblocks / 2) whose clusters, one per output tile, are all resident in a
// single wave; 1 when the tiles alone fill the GPU.
int tc_pick_splits(int M, int N, int K, int q4) {
  int bn = 16, lg = 0;
  while (bn < N && bn < 256) {
    bn *= 2;
    ++lg;
  }
  const long long tiles = (long long)((M + 127) / 128) * ((N + bn - 1) / bn);
  const int kblocks = (K + 63) / 64;
  int best = 1;
  for (int cz = 2; cz <= 8 && cz <= kblocks / 2; ++cz)
    if (tiles <= (q4 && lg < 2 ? g_max_clusters_q4[lg][cz] : g_max_clusters[lg][cz])) best = cz;
  return best;
}

cudaError_t launch_gemm_tc(const void* A, long long lda, int M, const void* B, long long ldb, int N,
                           int K, int swap, int splits, int32_t* err, const Epi& epi,
                           cudaStream_t st, int* launches, const void* a_tiles,
                           int late_trigger, int a_group_mtiles, int q4, int independent) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (q4 && (!a_tiles || !swap || N > 32)) return cudaErrorInvalidValue;
  int bn = 16;
  while (bn < N && bn < 256) bn *= 2;
  const int m_tiles = (M + 127) / 128;
  const int n_tiles = (N + bn - 1) / bn;
  TcArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.kblocks = (K + 63) / 64;
  a.swap = swap;
  a.prefetch_a = swap;
  a.err = err;
  a.splits = std::max(1, std::min(std::min(splits, 8), a.kblocks));
  a.a_tiles = static_cast<const uint8_t*>(a_tiles);
  a.late_trigger = late_trigger;
  a.independent = independent;
  a.mt0 = m_tiles;
  a.a_gm0 = a.a_gm1 = a_group_mtiles > 0 ? a_group_mtiles : m_tiles;
  CUtensorMap ma, mb;
  cudaError_t e = make_map(&mb, B, N, K, ldb, bn);
  if (e != cudaSuccess) return e;
  if (a_tiles)
    ma = mb;  // unused by the kernel
  else if ((e = make_map(&ma, A, M, K, lda, 128)) != cudaSuccess)
    return e;
  if (m_tiles > 65535 || n_tiles > 65535) return cudaErrorInvalidValue;
  dim3 grid(a.splits, m_tiles, n_tiles);
  ++*launches;
  if (q4) return launch_bn_q4(bn, ma, mb, mb, a, epi, epi, grid, st);
  return launch_bn(bn, ma, mb, mb, a, epi, epi, grid, st);
}

cudaError_t launch_gemm_tc_grouped(const void* a_tiles0, int M0, int gm0, const void* B0,
                                   long long ldb0, int N0, const Epi& epi0, const void* a_tiles1,
                                   int M1, const void* B1, long long ldb1, int N1, const Epi& epi1,
                                   int K, int splits, int32_t* err, cudaStream_t st, int* launches,
                                   int late_trigger, int q4) {
  if (M0 <= 0 || N0 <= 0 || M1 <= 0 || N1 <= 0 || !a_tiles0 || !a_tiles1)
    return cudaErrorInvalidValue;
  if (q4 && std::max(N0, N1) > 32) return cudaErrorInvalidValue;
  const int nmax = N0 > N1 ? N0 : N1;
  int bn = 16;
  while (bn < nmax && bn < 256) bn *= 2;
  const int mt0 = (M0 + 127) / 128, mt1 = (M1 + 127) / 128;
  const int n_tiles = (nmax + bn - 1) / bn;
  TcArgs a{};
  a.M = M0;
  a.N = N0;
  a.K = K;
  a.kblocks = (K + 63) / 64;
  a.swap = 1;
  a.prefetch_a = 1;
  a.err = err;
  a.splits = std::max(1, std::min(std::min(splits, 8), a.kblocks));
  a.a_tiles = static_cast<const uint8_t*>(a_tiles0);
  a.late_trigger = late_trigger;
  a.mt0 = mt0;
  a.M1 = M1;
  a.N1 = N1;
  a.a_tiles1 = static_cast<const uint8_t*>(a_tiles1);
  a.a_gm0 = gm0 > 0 ? gm0 : mt0;
  a.a_gm1 = mt1;
  CUtensorMap mb0, mb1;
  cudaError_t e = make_map(&mb0, B0, N0, K, ldb0, bn);
  if (e == cudaSuccess) e = make_map(&mb1, B1, N1, K, ldb1, bn);
  if (e != cudaSuccess) return e;
  if (mt0 + mt1 > 65535 || n_tiles > 65535) return cudaErrorInvalidValue;
  dim3 grid(a.splits, mt0 + mt1, n_tiles);
  ++*launches;
  if (q4) return launch_bn_q4(bn, mb0, mb0, mb1, a, epi0, epi1, grid, st);
  return launch_bn(bn, mb0, mb0, mb1, a, epi0, epi1, grid, st);
}

// Re-lay a row-major bf16 matrix [M][K] (host) as 128 x 64 tiles in the
// shared-memory image the kernel's tensor-core descriptors expect (rows of
// 128 bytes, 16-byte chunk c of row r at chunk c ^ (r & 7)), ordered
// [k_block][m_tile]; rows past M and columns past K are zero. CTAs walk their
// k-blocks in step, so at any moment the CTAs of a launch read one
// contiguous run of tiles (one k-block of every m-tile).
void tile_weights(const uint16_t* src, long long M, long long K, uint16_t* dst) {
  const long long mt = (M + 127) / 128, kb = (K + 63) / 64;
  for (long long t = 0; t < mt; ++t)
    for (long long b = 0; b < kb; ++b) {
      uint16_t* tile = dst + (b * mt + t) * 128 * 64;
      for (int r = 0; r < 128; ++r)
        for (int c = 0; c < 64; ++c) {
          const long long gr = t * 128 + r, gc = b * 64 + c;
          const uint16_t v = (gr < M && gc < K) ? src[gr * K + gc] : 0;
          tile[r * 64 + ((((c >> 3) ^ (r & 7))) << 3) + (c & 7)] = v;
        }
    }
}

size_t tiled_bytes(long long M, long long K) {
  return (size_t)((M + 127) / 128) * ((K + 63) / 64) * 128 * 64 * 2;
}

size_t q4_tiled_bytes(long long M, long long K) {
  return (size_t)((M + 127) / 128) * ((K + 63) / 64) * Q4_TILE_BYTES;
}

void tile_weights_q4(const uint8_t* codes, const uint32_t* prm, long long M, long long K,
                     uint8_t* dst) {
  const long long mt = (M + 127) / 128, kb = (K + 63) / 64, ng = (K + 127) / 128;
  for (long long t = 0; t < mt; ++t)
    for (long long b = 0; b < kb; ++b) {
      uint8_t* tile = dst + (size_t)(b * mt + t) * Q4_TILE_BYTES;
      for (int r = 0; r < 128; ++r) {
        const long long gr = t * 128 + r;
        // per 8 columns one 32-bit word; nibble i holds column 2i (i < 4) or
        // 2(i - 4) + 1, so that the kernel's pair j = nibbles (j, j + 4)
        for (int c = 0; c < 8; ++c) {
          uint32_t w = 0;
          for (int i = 0; i < 8; ++i) {
            const int e = i < 4 ? 2 * i : 2 * (i - 4) + 1;
            const long long gc = b * 64 + 8 * c + e;
            const uint32_t q = (gr < M && gc < K) ? codes[gr * K + gc] & 15u : 0u;
            w |= q << (4 * i);
          }
          std::memcpy(tile + r * 32 + 4 * c, &w, 4);
        }
        const uint32_t w = gr < M ? prm[gr * ng + (b * 64) / 128] : 0u;
        std::memcpy(tile + 4096 + r * 4, &w, 4);
      }
    }
}

}  // namespace hf
