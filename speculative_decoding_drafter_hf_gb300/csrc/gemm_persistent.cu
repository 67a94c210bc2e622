// Persistent, warp-specialised bf16 GEMM for the large token-major products
// of the prefill (tokens x features): D[m, n] = sum_k A[m, k] * B[n, k].
//
// One CTA per SM walks the output tiles t = blockIdx.x, + gridDim.x, ...
// (tile = 128 tokens x BN features) in grouped order: the token tiles come
// in groups whose rows fit well inside L2 (~48 MB), and within a group the
// tiles run feature-panel by feature-panel, so a wave of CTAs shares one or
// two weight panels and the group's token rows stay resident: every weight
// panel is read from DRAM once per group instead of once per wave. Warp 0 (one lane) feeds a ring of STAGES
// shared-memory slots with TMA, warp 1 (one lane) issues tcgen05.mma into
// one of two TMEM accumulators, and warps 2-5 drain the other accumulator
// through the epilogue, so a tile's epilogue overlaps the next tile's main
// loop. Every mbarrier wait is bounded; on expiry the kernel raises
// ERR_TIMEOUT, stops issuing work, drains its copies (bounded), frees TMEM
// and returns.
#include "common.cuh"
#include "tcgen05.cuh"

namespace hf {
namespace {

constexpr int PBN = 256;     // features per tile
constexpr int PSTAGES = 4;   // 4 x (16 KB A + 32 KB B)
constexpr int PTHREADS = 192;

struct PArgs {
  int M, N, K, kblocks, m_tiles, n_tiles;
  int group_m;  // token tiles per group of the tile order
  int32_t* err;
};

// Tile t of the grouped order -> (token tile mt, feature tile nt).
__device__ __forceinline__ void p_tile(const PArgs& a, int t, int& mt, int& nt) {
  const int per_group = a.group_m * a.n_tiles;
  const int g = t / per_group, local = t - g * per_group;
  const int g0 = g * a.group_m;
  const int gsz = a.m_tiles - g0 < a.group_m ? a.m_tiles - g0 : a.group_m;
  nt = local / gsz;
  mt = g0 + local % gsz;
}

constexpr size_t p_smem() {
  return 1024 + (size_t)PSTAGES * (128 * 128 + PBN * 128) + (2 * PSTAGES + 4) * 8 + 32;
}

__global__ void __launch_bounds__(PTHREADS, 1)
tc_gemm_persistent_kernel(const __grid_constant__ CUtensorMap ta,
                          const __grid_constant__ CUtensorMap tb, PArgs a, Epi epi) {
  constexpr int A_BYTES = 128 * 128, B_BYTES = PBN * 128;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t NCOLS = 2 * PBN;  // two accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + PSTAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + PSTAGES * B_BYTES);
  uint64_t* empty = full + PSTAGES;
  uint64_t* tfull = empty + PSTAGES;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;        // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] issued, [2] consumed

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int ntiles = a.m_tiles * a.n_tiles;
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    flags[0] = flags[1] = flags[2] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, NCOLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer over (tile, k-block), k-blocks numbered across tiles
    pdl_wait();
    int g = 0;
    for (int t = blockIdx.x; t < ntiles && !*(volatile int*)&flags[0]; t += gridDim.x) {
      int mt, nt;
      p_tile(a, t, mt, nt);
      for (int kb = 0; kb < a.kblocks; ++kb, ++g) {
        const int s = g % PSTAGES;
        const uint32_t ph = (uint32_t)(g / PSTAGES) & 1u;
        if (g >= PSTAGES && !mbar_wait(&empty[s], ph ^ 1u)) {
          atomicExch(&flags[0], 1);
          break;
        }
        mbar_expect_tx(&full[s], STAGE_BYTES);
        tma_load_2d(sA + s * A_BYTES, &ta, &full[s], kb * 64, mt * 128);
        tma_load_2d(sB + s * B_BYTES, &tb, &full[s], kb * 64, nt * PBN);
      }
    }
    flags[1] = g;
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: accumulator buffer i % 2 for the i-th tile of this CTA
    constexpr uint32_t idesc = idesc_bf16(PBN);
    int g = 0, i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++i) {
      const int buf = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      if (!mbar_wait(&tempty[buf], aph ^ 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * PBN);
      for (int kb = 0; kb < a.kblocks; ++kb, ++g) {
        const int s = g % PSTAGES;
        const uint32_t ph = (uint32_t)(g / PSTAGES) & 1u;
        if (!mbar_wait(&full[s], ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = sdesc_sw128(sA + s * A_BYTES);
        const uint64_t db = sdesc_sw128(sB + s * B_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(acc, da + 2ull * kk, db + 2ull * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&empty[s]);
      }
      if (!ok) break;
      umma_commit(&tfull[buf]);
    }
    if (!ok) atomicExch(&flags[0], 1);
    flags[2] = g;
  } else if (warp >= 2) {
    // Epilogue: TMEM lane quadrant (warp % 4) holds tile rows 32*(warp%4) + lane
    pdl_wait();
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      const uint32_t aph = (uint32_t)(i >> 1) & 1u;
      int mt, nt;
      p_tile(a, t, mt, nt);
      const int m = mt * 128 + quad * 32 + lane;
      // the commit epilogue's per-row part (request, position: dependent
      // global loads) once per tile row, issued before the accumulator wait
      const bool kv = epi.kind == EPI_SSM_KV;
      const long long ro = kv && m < a.M ? ssm_kv_row(epi, m, nt * PBN) : -1;
      if (!mbar_wait(&tfull[buf], aph)) {
        atomicExch(&flags[0], 1);
        break;
      }
      tc_fence_after();
      float v[16];
#pragma unroll 1
      for (int c0 = 0; c0 < PBN; c0 += 16) {
        tmem_ld16(tmem + lane_base + (uint32_t)(buf * PBN + c0), v);
        const int n0 = nt * PBN + c0;
        if (m < a.M && n0 < a.N) {
          if (kv)
            epi_ssm_chunk16(epi, m, n0, min(16, a.N - n0), v, ro);
          else
            epi_chunk16(epi, m, n0, min(16, a.N - n0), v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[buf])) : "memory");
    }
  }
  __syncwarp();
  __syncthreads();
  if (flags[0]) {
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      for (int g = flags[2]; g < flags[1]; ++g)
        mbar_wait(&full[g % PSTAGES], (uint32_t)(g / PSTAGES) & 1u);  // bounded drain
    }
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, NCOLS);
}

}  // namespace

cudaError_t configure_tc_persistent(int num_sms) {
  (void)num_sms;
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_persistent_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p_smem());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_persistent_kernel,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t launch_gemm_persistent(const void* A, long long lda, int M, const void* B,
                                   long long ldb, int N, int K, int32_t* err, const Epi& epi,
                                   int num_sms, cudaStream_t st, int* launches) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  PArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.kblocks = (K + 63) / 64;
  a.m_tiles = (M + 127) / 128;
  a.n_tiles = (N + PBN - 1) / PBN;
  // token tiles per group: their rows (128 x K bf16 each) within ~48 MB of L2
  a.group_m = (int)std::max<long long>(1, std::min<long long>(a.m_tiles, (48ll << 20) / (256ll * K)));
  a.err = err;
  CUtensorMap ma, mb;
  cudaError_t e = make_map(&ma, A, M, K, lda, 128);
  if (e == cudaSuccess) e = make_map(&mb, B, N, K, ldb, PBN);
  if (e != cudaSuccess) return e;
  const int tiles = a.m_tiles * a.n_tiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  ++*launches;
  return launch_pdl(tc_gemm_persistent_kernel, dim3(grid), dim3(PTHREADS), p_smem(), st, ma, mb,
                    a, epi);
}

}  // namespace hf
