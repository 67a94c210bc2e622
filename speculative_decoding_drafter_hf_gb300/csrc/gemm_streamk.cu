// Stream-K tcgen05 GEMM for the skinny swapped products (weights x a few
// activation rows): D[m, n] = sum_k A[m, k] * B[n, k] with A pre-tiled
// weights (tile_weights), B at most 32 activation rows (one n-tile), output
// row n, column m. One or two products (same K) per launch.
//
// The work -- every (m-tile, k-block) unit of both products -- is split into
// equal contiguous shares, one per CTA, one CTA per SM: every SM streams the
// same number of weight tiles whatever the tile count (no partial last wave,
// no idle SMs when the tiles are fewer than the SMs). A CTA's share covers
// parts of one or more tiles ("segments"). A segment that is a whole tile
// goes straight through the epilogue; otherwise its partial accumulator is
// written to a workspace slot, and the CTA that completes a tile's last
// segment (ticket per tile) sums the tile's slots in k order -- deterministic,
// whichever CTA arrives last -- runs the epilogue and resets the ticket.
//
// Warp 0 (one lane) streams A tiles (bulk copies) and B tiles (TMA) through a
// ring of STAGES slots; warp 1 (one lane) issues tcgen05.mma into one of two
// TMEM accumulators (alternating per segment); warps 2-5 drain the other
// accumulator (epilogue or partial), so a segment's epilogue overlaps the
// next segment's main loop. Every wait is bounded; on expiry the kernel
// raises ERR_TIMEOUT, stops, drains its copies (bounded), frees TMEM.
#include "common.cuh"
#include "tcgen05.cuh"

namespace hf {
namespace {

constexpr int SK_THREADS = 192;

struct SkArgs {
  int kblocks;
  int mt0, mt1;       // m-tiles of each product (mt1 = 0: one product)
  int M0, N0, M1, N1;
  int gm0, gm1;       // m-tiles per stored group of the tiled A (see launch_gemm_tc)
  const uint8_t* at0;
  const uint8_t* at1;
  long long U;        // units = (mt0 + mt1) * kblocks
  int G;              // CTAs
  int nslot;          // workspace slots per tile
  float* ws;          // [tile][slot][BN][128] partial accumulators
  int* tickets;       // [tile], zero between launches
  int late_trigger;
  int32_t* err;
};

__host__ __device__ inline long long sk_start(long long g, long long U, int G) {
  return g * U / G;
}
// CTA whose share holds unit x: the largest g with floor(g U / G) <= x.
__host__ __device__ inline int sk_owner(long long x, long long U, int G) {
  return (int)(((x + 1) * G - 1) / U);
}

template <int BN, int STAGES>
constexpr size_t sk_smem() {
  // alignment slack, stages, barriers (full, empty, tfull[2], tempty[2]),
  // TMEM slot + flags, per-row epilogue cache of both products
  return 1024 + (size_t)STAGES * (128 * 128 + BN * 128) + (2 * STAGES + 4) * 8 + 32 +
         2 * BN * 8 + 16;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(SK_THREADS, 1)
tc_gemm_sk_kernel(const __grid_constant__ CUtensorMap tb0, const __grid_constant__ CUtensorMap tb1,
                  SkArgs a, const __grid_constant__ Epi epi0, const __grid_constant__ Epi epi1) {
  constexpr int A_BYTES = 128 * 128, B_BYTES = BN * 128;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t NCOLS = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2] accumulator ready
  uint64_t* tempty = tfull + 2;      // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] issued, [2] consumed, [3] last
  long long* ep_ro = reinterpret_cast<long long*>(flags + 7);  // [2][BN] ring-row offsets (8-aligned)

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = blockIdx.x;
  const int kb = a.kblocks;
  const long long u0 = sk_start(g, a.U, a.G), u1 = sk_start(g + 1, a.U, a.G);
  const int nu = (int)(u1 - u0);
  if (!a.late_trigger) pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    flags[0] = flags[1] = flags[2] = flags[3] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, NCOLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // producer over this CTA's units
    auto load_a = [&](int s, long long u) {
      const int t = (int)(u / kb), k = (int)(u % kb);
      const bool second = t >= a.mt0;
      const int mt = second ? t - a.mt0 : t;
      const int gm = second ? a.gm1 : a.gm0;
      const uint8_t* at = second ? a.at1 : a.at0;
      const size_t idx = ((size_t)(mt / gm) * kb + k) * gm + mt % gm;
      bulk_g2s(sA + s * A_BYTES, at + idx * (size_t)A_BYTES, A_BYTES, &full[s]);
    };
    auto load_b = [&](int s, long long u) {
      const int t = (int)(u / kb), k = (int)(u % kb);
      tma_load_2d(sB + s * B_BYTES, t >= a.mt0 ? &tb1 : &tb0, &full[s], k * 64, 0);
    };
    const int pre = nu < STAGES ? nu : STAGES;
    for (int j = 0; j < pre; ++j) {  // weights do not depend on earlier launches
      mbar_expect_tx(&full[j], STAGE_BYTES);
      load_a(j, u0 + j);
    }
    pdl_wait();
    if (a.late_trigger) pdl_trigger();
    for (int j = 0; j < pre; ++j) load_b(j, u0 + j);
    int i = pre;
    for (; i < nu; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u)) {
        atomicExch(&flags[0], 1);
        break;
      }
      if (*(volatile int*)&flags[0]) break;
      mbar_expect_tx(&full[s], STAGE_BYTES);
      load_a(s, u0 + i);
      load_b(s, u0 + i);
    }
    flags[1] = i;
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: segment j of this CTA accumulates into buffer j % 2
    if (a.late_trigger) {
      pdl_wait();
      pdl_trigger();
    }
    constexpr uint32_t idesc = idesc_bf16(BN);
    int i = 0, j = 0;
    bool ok = true;
    while (i < nu && ok) {
      const long long u = u0 + i;
      const int t = (int)(u / kb);
      const int seg_end = (int)(min(u1, (long long)(t + 1) * kb) - u0);  // exclusive, local
      const int buf = j & 1;
      if (!mbar_wait(&tempty[buf], ((uint32_t)(j >> 1) & 1u) ^ 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * BN);
      const int first = i;
      for (; i < seg_end; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&full[s], (uint32_t)(i / STAGES) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = sdesc_sw128(sA + s * A_BYTES);
        const uint64_t db = sdesc_sw128(sB + s * B_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(acc, da + 2ull * kk, db + 2ull * kk, idesc, (i > first || kk > 0) ? 1u : 0u);
        umma_commit(&empty[s]);
      }
      if (!ok) break;
      umma_commit(&tfull[buf]);
      ++j;
    }
    if (!ok) atomicExch(&flags[0], 1);
    flags[2] = i;
  } else if (warp >= 2) {
    // epilogue warps: TMEM lane quadrant warp % 4 holds tile rows 32*(warp%4) + lane
    const int quad = warp & 3;
    const int et = tid - 64;  // 0..127
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    pdl_wait();  // the epilogue reads activations' row data and writes outputs
    if (a.late_trigger) pdl_trigger();
    // per-row data of the ring append (rows are the same for every tile)
    for (int e = et; e < 2 * BN; e += 128) {
      const int p = e / BN, n = e % BN;
      const Epi& ep = p ? epi1 : epi0;
      long long ro = -1;
      if (ep.kind == EPI_SSM_KV && n < (p ? a.N1 : a.N0)) {
        int bq;
        long long pq;
        epi_row(ep, n, bq, pq, 0);
        ro = ssm_row_off(ep.d, bq, pq);
      }
      ep_ro[e] = ro;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    int i = 0, j = 0;
    while (i < nu) {
      const long long u = u0 + i;
      const int t = (int)(u / kb);
      const long long t_lo = (long long)t * kb, t_hi = t_lo + kb;
      const int seg_end = (int)(min(u1, t_hi) - u0);
      i = seg_end;
      const int buf = j & 1;
      if (!mbar_wait(&tfull[buf], (uint32_t)(j >> 1) & 1u)) {
        atomicExch(&flags[0], 1);
        break;
      }
      ++j;
      tc_fence_after();
      float v[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) tmem_ld16(tmem + lane_base + (uint32_t)(buf * BN + c0), v + c0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[buf])) : "memory");

      const bool second = t >= a.mt0;
      const int mt = second ? t - a.mt0 : t;
      const int M = second ? a.M1 : a.M0, N = second ? a.N1 : a.N0;
      const Epi& ep = second ? epi1 : epi0;
      const int m = mt * 128 + quad * 32 + lane;
      const int gfirst = sk_owner(t_lo, a.U, a.G), glast = sk_owner(t_hi - 1, a.U, a.G);
      const int nseg = glast - gfirst + 1;
      if (nseg > 1) {
        // partial: slot g - gfirst of tile t; the last segment to arrive sums them
        float* slot = a.ws + ((size_t)t * a.nslot + (g - gfirst)) * (BN * 128);
#pragma unroll
        for (int n = 0; n < BN; ++n) slot[n * 128 + et] = v[n];
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (et == 0) flags[3] = atomicAdd(&a.tickets[t], 1) == nseg - 1;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const bool last = flags[3] != 0;
        asm volatile("bar.sync 1, 128;" ::: "memory");  // flag read before the next segment
        if (!last) continue;
        __threadfence();
        const float* base = a.ws + (size_t)t * a.nslot * (BN * 128);
#pragma unroll
        for (int n = 0; n < BN; ++n) v[n] = 0.f;
        for (int q = 0; q < nseg; ++q)
#pragma unroll
          for (int n = 0; n < BN; ++n) v[n] += __ldcg(base + (size_t)q * BN * 128 + n * 128 + et);
        if (et == 0) a.tickets[t] = 0;  // ready for the next launch
      }
      if (m >= M) continue;
      // epilogue: output row n, column m
      if (ep.kind == EPI_F32) {
#pragma unroll
        for (int n = 0; n < BN; ++n)
          if (n < N) ep.out[(size_t)n * ep.ld + m] = v[n];
      } else if (ep.kind == EPI_RESID) {
        const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(ep.resid);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ep.out_t);
        float x[BN];
#pragma unroll
        for (int n = 0; n < BN; ++n) x[n] = n < N ? to_f(__ldcg(&res[(size_t)n * ep.ld + m])) : 0.f;
#pragma unroll
        for (int n = 0; n < BN; ++n)
          if (n < N) out[(size_t)n * ep.ld + m] = __float2bfloat16_rn(x[n] + v[n]);
      } else if (ep.kind == EPI_SSM_KV) {
        const SsmCol col = ssm_col(ep, m);
        const long long* ro = ep_ro + (second ? BN : 0);
#pragma unroll
        for (int n = 0; n < BN; ++n)
          if (n < N) ssm_store<__nv_bfloat16>(ep, col, n, ro[n], v[n]);
      }
    }
  } else if (a.late_trigger) {
    pdl_wait();
    pdl_trigger();
  }
  __syncwarp();
  __syncthreads();
  if (flags[0]) {
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      for (int i = flags[2]; i < flags[1]; ++i)
        mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u);  // bounded drain
    }
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, NCOLS);
}

constexpr int SK_STAGES16 = 8, SK_STAGES32 = 7;

template <int BN, int STAGES>
cudaError_t sk_configure() {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_sk_kernel<BN, STAGES>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sk_smem<BN, STAGES>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_sk_kernel<BN, STAGES>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

template <int BN, int STAGES>
cudaError_t sk_launch(const CUtensorMap& mb0, const CUtensorMap& mb1, const SkArgs& a,
                      const Epi& epi0, const Epi& epi1, cudaStream_t st) {
  return launch_pdl(tc_gemm_sk_kernel<BN, STAGES>, dim3(a.G), dim3(SK_THREADS),
                    sk_smem<BN, STAGES>(), st, mb0, mb1, a, epi0, epi1);
}

}  // namespace

cudaError_t configure_gemm_sk() {
  cudaError_t e = sk_configure<16, SK_STAGES16>();
  if (e == cudaSuccess) e = sk_configure<32, SK_STAGES32>();
  return e;
}

size_t gemm_sk_workspace(int M0, int M1, int K, int num_sms, int* tiles, int* nslot) {
  const int kb = (K + 63) / 64;
  const int mt = (M0 + 127) / 128 + (M1 > 0 ? (M1 + 127) / 128 : 0);
  const long long U = (long long)mt * kb;
  const int G = (int)std::min<long long>(num_sms, U);
  int worst = 1;
  for (int t = 0; t < mt; ++t) {
    const int n = sk_owner((long long)(t + 1) * kb - 1, U, G) - sk_owner((long long)t * kb, U, G) + 1;
    worst = std::max(worst, n);
  }
  *tiles = mt;
  *nslot = worst;
  return (size_t)mt * worst * 32 * 128;  // floats, for the widest tile (BN = 32)
}

cudaError_t launch_gemm_sk(const void* a_tiles0, int M0, int gm0, const void* B0, long long ldb0,
                           int N0, const Epi& epi0, const void* a_tiles1, int M1, const void* B1,
                           long long ldb1, int N1, const Epi& epi1, int K, int num_sms, float* ws,
                           size_t ws_floats, int* tickets, int n_tickets, int32_t* err,
                           int late_trigger, cudaStream_t st, int* launches) {
  const bool two = a_tiles1 != nullptr && M1 > 0 && N1 > 0;
  const int nmax = std::max(N0, two ? N1 : 0);
  if (M0 <= 0 || N0 <= 0 || nmax > 32 || !a_tiles0) return cudaErrorInvalidValue;
  const int bn = nmax <= 16 ? 16 : 32;
  int tiles = 0, nslot = 0;
  const size_t need = gemm_sk_workspace(M0, two ? M1 : 0, K, num_sms, &tiles, &nslot);
  if (need > ws_floats || tiles > n_tickets) return cudaErrorInvalidValue;
  SkArgs a{};
  a.kblocks = (K + 63) / 64;
  a.mt0 = (M0 + 127) / 128;
  a.mt1 = two ? (M1 + 127) / 128 : 0;
  a.M0 = M0;
  a.N0 = N0;
  a.M1 = two ? M1 : 0;
  a.N1 = two ? N1 : 0;
  a.gm0 = gm0 > 0 ? gm0 : a.mt0;
  a.gm1 = a.mt1 > 0 ? a.mt1 : 1;
  a.at0 = static_cast<const uint8_t*>(a_tiles0);
  a.at1 = static_cast<const uint8_t*>(two ? a_tiles1 : a_tiles0);
  a.U = (long long)(a.mt0 + a.mt1) * a.kblocks;
  a.G = (int)std::min<long long>(num_sms, a.U);
  a.nslot = nslot;
  a.ws = ws;
  a.tickets = tickets;
  a.late_trigger = late_trigger;
  a.err = err;
  CUtensorMap mb0, mb1;
  cudaError_t e = make_map(&mb0, B0, N0, K, ldb0, bn);
  if (e == cudaSuccess) e = two ? make_map(&mb1, B1, N1, K, ldb1, bn) : cudaSuccess;
  if (e != cudaSuccess) return e;
  if (!two) mb1 = mb0;
  ++*launches;
  return bn == 16 ? sk_launch<16, SK_STAGES16>(mb0, mb1, a, epi0, two ? epi1 : epi0, st)
                  : sk_launch<32, SK_STAGES32>(mb0, mb1, a, epi0, two ? epi1 : epi0, st);
}

}  // namespace hf
