// Token-major stream-K tcgen05 GEMM for the wide activation x weight products
// (more than 32 activation rows, i.e. batches of 5+ requests):
// D[m, n] = sum_k X[m, k] * W[n, k] with X the activation rows (tokens) and W
// the weights in their plain K-major layout, both through TMA; output row m
// (token), column n (feature). One or two products (same K) per launch.
//
// Tiles are 128 tokens x 256 features; the work -- every (token tile,
// feature tile, k-block) unit of both products -- is split into equal shares,
// one per CTA, one CTA per SM (tokens innermost, so the CTAs working on one
// weight panel run side by side and share it in L2). A CTA's share covers
// parts of one or more tiles ("segments"); only its first and last can be
// partial. A whole tile goes straight through the epilogue; a partial
// segment's accumulator goes to the CTA's workspace slot (two per CTA), and
// the CTA completing a tile's last segment (ticket per tile) sums the tile's
// slots in k order -- deterministic whichever CTA arrives last -- runs the
// epilogue and resets the ticket. In this orientation a thread's accumulator
// row is one token and its 16-column chunks are 16 consecutive features, so
// the epilogue moves contiguous runs (epi_chunk16).
//
// With at least as many tiles as CTAs the launch is data-parallel instead
// (dp): CTA g takes whole tiles g, g + G, g + 2G, ...; with tokens innermost
// the CTAs 4s..4s+3 of a wave then stream the same weight panel at the same
// time (one DRAM read, the other three from L2), where contiguous stream-K
// shares would come back to a panel only after a whole tile of every CTA.
//
// Warp 0 (one lane) streams W (before the dependency wait: weights do not
// depend on earlier launches) and X through a ring of STAGES slots; warp 1
// (one lane) issues tcgen05.mma into one of two TMEM accumulators; warps 2-9
// drain the other one, warps 2-5 the first 128 columns and warps 6-9 the last
// 128 (the epilogue is latency-bound: two groups halve its chain). Every wait
// is bounded; on expiry the kernel raises ERR_TIMEOUT, stops, drains its
// copies (bounded) and frees TMEM.
#include "common.cuh"
#include "tcgen05.cuh"

namespace hf {
namespace {

constexpr int TM_THREADS = 320;  // producer, MMA, two groups of 4 epilogue warps
constexpr int TM_BN = 256;     // features per tile
constexpr int TM_STAGES = 4;   // 4 x (16 KB tokens + 32 KB weights)

struct TmArgs {
  int kblocks;
  int mt0, nt0, mt1, nt1;  // token tiles, feature tiles of each product (mt1 = 0: one product)
  int M0, N0, M1, N1;      // tokens, features
  long long U;             // units
  int G;                   // CTAs
  float* ws;               // [2G][16 chunks][128][16] partial slots
  int* tickets;            // [tile], zero between launches
  int late_trigger;        // 1: signal dependents only after the dependency wait
  int dp;                  // 1: whole tiles g, g + G, ... per CTA (no partial tiles)
  int tiles;               // tiles of both products
  int32_t* err;
};

__host__ __device__ inline long long tm_start(long long g, long long U, int G) { return g * U / G; }
__host__ __device__ inline int tm_owner(long long x, long long U, int G) {
  return (int)(((x + 1) * G - 1) / U);
}

constexpr size_t tm_smem() {
  return 1024 + (size_t)TM_STAGES * (128 * 128 + TM_BN * 128) + (2 * TM_STAGES + 4) * 8 + 32;
}

__global__ void __launch_bounds__(TM_THREADS, 1)
tc_gemm_tm_kernel(const __grid_constant__ CUtensorMap tx0, const __grid_constant__ CUtensorMap tw0,
                  const __grid_constant__ CUtensorMap tx1, const __grid_constant__ CUtensorMap tw1,
                  TmArgs a, const __grid_constant__ Epi epi0, const __grid_constant__ Epi epi1) {
  constexpr int X_BYTES = 128 * 128, W_BYTES = TM_BN * 128;
  constexpr uint32_t STAGE_BYTES = X_BYTES + W_BYTES;
  constexpr uint32_t NCOLS = 2 * TM_BN;  // two accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sX = smem;
  uint8_t* sW = smem + TM_STAGES * X_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sW + TM_STAGES * W_BYTES);
  uint64_t* empty = full + TM_STAGES;
  uint64_t* tfull = empty + TM_STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] issued, [2] consumed, [3] last

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = blockIdx.x;
  const int kb = a.kblocks;
  const int T0 = a.mt0 * a.nt0;
  const long long u0 = a.dp ? 0 : tm_start(g, a.U, a.G), u1 = a.dp ? 0 : tm_start(g + 1, a.U, a.G);
  const int nu = a.dp ? (g < a.tiles ? (a.tiles - 1 - g) / a.G + 1 : 0) * kb : (int)(u1 - u0);
  const int first_tile = (int)(u0 / kb);
  // global unit of this CTA's i-th unit, and the end (local) of the segment holding it
  auto gu = [&](int i) -> long long {
    return a.dp ? (long long)(g + (i / kb) * a.G) * kb + i % kb : u0 + i;
  };
  auto seg_end_of = [&](int i) -> int {
    if (a.dp) return (i / kb + 1) * kb;
    const long long t = (u0 + i) / kb;
    return (int)(min(u1, (t + 1) * kb) - u0);
  };
  // tile t -> product, token tile, feature tile (token tiles innermost)
  auto tile_of = [&](int t, bool& second, int& mt, int& nt) {
    second = t >= T0;
    const int tl = second ? t - T0 : t;
    const int mtp = second ? a.mt1 : a.mt0;
    mt = tl % mtp;
    nt = tl / mtp;
  };
  if (!a.late_trigger) pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < TM_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // one arrival per epilogue warp
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
    auto load_w = [&](int s, long long u) {
      bool second;
      int mt, nt;
      tile_of((int)(u / kb), second, mt, nt);
      tma_load_2d(sW + s * W_BYTES, second ? &tw1 : &tw0, &full[s], (int)(u % kb) * 64, nt * TM_BN);
    };
    auto load_x = [&](int s, long long u) {
      bool second;
      int mt, nt;
      tile_of((int)(u / kb), second, mt, nt);
      tma_load_2d(sX + s * X_BYTES, second ? &tx1 : &tx0, &full[s], (int)(u % kb) * 64, mt * 128);
    };
    const int pre = nu < TM_STAGES ? nu : TM_STAGES;
    for (int j = 0; j < pre; ++j) {
      mbar_expect_tx(&full[j], STAGE_BYTES);
      load_w(j, gu(j));
    }
    pdl_wait();
    if (a.late_trigger) pdl_trigger();
    for (int j = 0; j < pre; ++j) load_x(j, gu(j));
    int i = pre;
    for (; i < nu; ++i) {
      const int s = i % TM_STAGES;
      const uint32_t ph = (uint32_t)(i / TM_STAGES) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u)) {
        atomicExch(&flags[0], 1);
        break;
      }
      if (*(volatile int*)&flags[0]) break;
      mbar_expect_tx(&full[s], STAGE_BYTES);
      load_w(s, gu(i));
      load_x(s, gu(i));
    }
    flags[1] = i;
  } else if (warp == 1 && lane == 0) {
    if (a.late_trigger) {
      pdl_wait();
      pdl_trigger();
    }
    constexpr uint32_t idesc = idesc_bf16(TM_BN);
    int i = 0, j = 0;
    bool ok = true;
    while (i < nu && ok) {
      const int seg_end = seg_end_of(i);
      const int buf = j & 1;
      if (!mbar_wait(&tempty[buf], ((uint32_t)(j >> 1) & 1u) ^ 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * TM_BN);
      const int first = i;
      for (; i < seg_end; ++i) {
        const int s = i % TM_STAGES;
        if (!mbar_wait(&full[s], (uint32_t)(i / TM_STAGES) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = sdesc_sw128(sX + s * X_BYTES);
        const uint64_t db = sdesc_sw128(sW + s * W_BYTES);
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
    // epilogue: TMEM lane quadrant warp % 4 holds token rows 32*(warp%4) + lane;
    // group eg takes columns [128 eg, 128 eg + 128)
    const int quad = warp & 3;
    const int eg = (warp - 2) >> 2;
    const int cb = eg * (TM_BN / 2), ce = cb + TM_BN / 2;
    const int ml = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    pdl_wait();
    if (a.late_trigger) pdl_trigger();
    int i = 0, j = 0;
    while (i < nu) {
      const long long u = gu(i);
      const int t = (int)(u / kb);
      const long long t_lo = (long long)t * kb, t_hi = t_lo + kb;
      i = seg_end_of(i);
      const int buf = j & 1;
      if (!mbar_wait(&tfull[buf], (uint32_t)(j >> 1) & 1u)) {
        atomicExch(&flags[0], 1);
        break;
      }
      ++j;
      tc_fence_after();
      const uint32_t acc = tmem + lane_base + (uint32_t)(buf * TM_BN);
      bool second;
      int mt, nt;
      tile_of(t, second, mt, nt);
      const int M = second ? a.M1 : a.M0, N = second ? a.N1 : a.N0;
      const Epi& ep = second ? epi1 : epi0;
      const int m = mt * 128 + ml, n_base = nt * TM_BN;
      const int gfirst = a.dp ? g : tm_owner(t_lo, a.U, a.G);
      const int glast = a.dp ? g : tm_owner(t_hi - 1, a.U, a.G);
      const int nseg = glast - gfirst + 1;
      float v[16];
      if (nseg > 1) {
        // partial: [chunk][token][16] floats in this CTA's slot
        float* slot = a.ws + ((size_t)2 * g + (t > first_tile ? 1 : 0)) * (TM_BN * 128);
#pragma unroll 1
        for (int c0 = cb; c0 < ce; c0 += 16) {
          tmem_ld16(acc + (uint32_t)c0, v);
          float4* dst = reinterpret_cast<float4*>(slot + ((size_t)(c0 >> 4) * 128 + ml) * 16);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[buf])) : "memory");
        __threadfence();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (tid == 64) flags[3] = atomicAdd(&a.tickets[t], 1) == nseg - 1;
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const bool last = flags[3] != 0;
        asm volatile("bar.sync 1, 256;" ::: "memory");  // flag read before the next segment
        if (!last) continue;
        __threadfence();
#pragma unroll 1
        for (int c0 = cb; c0 < ce && n_base + c0 < N; c0 += 16) {
          // k order: CTA gfirst's slot (its last segment), the middle CTAs'
          // (their only one), glast's (its first)
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = 0.f;
          for (int h0 = gfirst; h0 <= glast; h0 += 4) {
            float4 r[4][4];
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              const int h = h0 + hh;
              if (h <= glast) {
                const int sidx = 2 * h + (h == gfirst && t > (int)(tm_start(h, a.U, a.G) / kb) ? 1 : 0);
                const float4* sp = reinterpret_cast<const float4*>(
                    a.ws + (size_t)sidx * (TM_BN * 128) + ((size_t)(c0 >> 4) * 128 + ml) * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) r[hh][q] = __ldcg(sp + q);
              }
            }
#pragma unroll
            for (int hh = 0; hh < 4; ++hh)
              if (h0 + hh <= glast)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  v[4 * q] += r[hh][q].x;
                  v[4 * q + 1] += r[hh][q].y;
                  v[4 * q + 2] += r[hh][q].z;
                  v[4 * q + 3] += r[hh][q].w;
                }
          }
          if (m < M) epi_chunk16(ep, m, n_base + c0, min(16, N - n_base - c0), v);
        }
        if (tid == 64) a.tickets[t] = 0;  // ready for the next launch
        continue;
      }
#pragma unroll 1
      for (int c0 = cb; c0 < ce; c0 += 16) {
        tmem_ld16(acc + (uint32_t)c0, v);
        if (m < M && n_base + c0 < N) epi_chunk16(ep, m, n_base + c0, min(16, N - n_base - c0), v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[buf])) : "memory");
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
        mbar_wait(&full[i % TM_STAGES], (uint32_t)(i / TM_STAGES) & 1u);  // bounded drain
    }
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, NCOLS);
}

}  // namespace

cudaError_t configure_gemm_tm() {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_tm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tm_smem());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_tm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

size_t gemm_tm_workspace(int num_sms) { return (size_t)2 * num_sms * TM_BN * 128; }

cudaError_t launch_gemm_tm(const void* X0, long long ldx0, int M0, const void* W0, long long ldw0,
                           int N0, const Epi& epi0, const void* X1, long long ldx1, int M1,
                           const void* W1, long long ldw1, int N1, const Epi& epi1, int K,
                           int num_sms, float* ws, size_t ws_floats, int* tickets, int n_tickets,
                           int32_t* err, int late_trigger, cudaStream_t st, int* launches) {
  const bool two = X1 != nullptr && W1 != nullptr && M1 > 0 && N1 > 0;
  if (M0 <= 0 || N0 <= 0) return cudaErrorInvalidValue;
  TmArgs a{};
  a.kblocks = (K + 63) / 64;
  a.mt0 = (M0 + 127) / 128;
  a.nt0 = (N0 + TM_BN - 1) / TM_BN;
  a.mt1 = two ? (M1 + 127) / 128 : 0;
  a.nt1 = two ? (N1 + TM_BN - 1) / TM_BN : 0;
  a.M0 = M0;
  a.N0 = N0;
  a.M1 = two ? M1 : 0;
  a.N1 = two ? N1 : 0;
  const long long tiles = (long long)a.mt0 * a.nt0 + (long long)a.mt1 * a.nt1;
  a.U = tiles * a.kblocks;
  a.G = (int)std::min<long long>(num_sms, a.U);
  a.tiles = (int)tiles;
  a.dp = tiles >= a.G ? 1 : 0;  // enough whole tiles for every CTA
  if (tiles > n_tickets || gemm_tm_workspace(a.G) > ws_floats) return cudaErrorInvalidValue;
  a.ws = ws;
  a.tickets = tickets;
  a.late_trigger = late_trigger;
  a.err = err;
  CUtensorMap mx0, mw0, mx1, mw1;
  cudaError_t e = make_map(&mx0, X0, M0, K, ldx0, 128);
  if (e == cudaSuccess) e = make_map(&mw0, W0, N0, K, ldw0, TM_BN);
  if (e == cudaSuccess && two) e = make_map(&mx1, X1, M1, K, ldx1, 128);
  if (e == cudaSuccess && two) e = make_map(&mw1, W1, N1, K, ldw1, TM_BN);
  if (e != cudaSuccess) return e;
  if (!two) {
    mx1 = mx0;
    mw1 = mw0;
  }
  ++*launches;
  return launch_pdl(tc_gemm_tm_kernel, dim3(a.G), dim3(TM_THREADS), tm_smem(), st, mx0, mw0, mx1,
                    mw1, a, epi0, two ? epi1 : epi0);
}

}  // namespace hf
