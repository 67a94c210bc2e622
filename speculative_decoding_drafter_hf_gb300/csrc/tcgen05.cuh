// tcgen05 / TMEM helpers shared by the tensor-core GEMM kernels (inline PTX).
#pragma once

#include "common.cuh"

namespace hf {

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile whose rows are 128 bytes
// (64 bf16) with the 128-byte swizzle; 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(const void* p) {
  const uint64_t a = smem_u32(p);
  uint64_t d = (a >> 4) & 0x3FFFull;   // start address
  d |= 1ull << 16;                     // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 B
  d |= 1ull << 46;                     // descriptor version
  d |= 2ull << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulate, both
// operands K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}


__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// Residual epilogue of 16 columns of row m (ld % 8 == 0) whose residual
// bf16 values r0 | r1 the caller has loaded: out = bf16(resid + v).
__device__ __forceinline__ void epi_resid16(const Epi& e, int m, int n0, const float* v, uint4 r0,
                                            uint4 r1) {
  uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(e.out_t) + (size_t)m * e.ld + n0);
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&r0);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&r1);
  uint4 w0, w1;
  __nv_bfloat162* c2 = reinterpret_cast<__nv_bfloat162*>(&w0);
  __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(&w1);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 fa = __bfloat1622float2(a2[q]), fb = __bfloat1622float2(b2[q]);
    c2[q] = __floats2bfloat162_rn(fa.x + v[2 * q], fa.y + v[2 * q + 1]);
    d2[q] = __floats2bfloat162_rn(fb.x + v[8 + 2 * q], fb.y + v[8 + 2 * q + 1]);
  }
  o[0] = w0;
  o[1] = w1;
}

// Commit-projection epilogue (EPI_SSM_KV) of 16 columns of row m whose
// ring-row offset ro the caller has computed (ssm_kv_row; -1: the row is
// skipped).
__device__ __forceinline__ void epi_ssm_chunk16(const Epi& e, int m, int n0, int ncols,
                                                const float* v, long long ro) {
  const Dims& d = e.d;
  if (ro < 0) return;
  // the 16 columns usually fall in one region (one ring head, or the x / B /
  // dt block): one column look-up and 16-byte stores then
  const SsmCol k0 = ssm_col(e, n0);
  if (ncols == 16) {
    const SsmCol k15 = ssm_col(e, n0 + 15);
    if (k0.kind == 1 && k15.kind == 1 && k15.ring == k0.ring && k15.base == k0.base + 15) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(k0.ring) + k0.base + ro;
      if ((reinterpret_cast<uintptr_t>(o) & 15) == 0) {
        uint4 w[2];
        __nv_bfloat162* w2 = reinterpret_cast<__nv_bfloat162*>(w);
#pragma unroll
        for (int q = 0; q < 8; ++q) w2[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
        reinterpret_cast<uint4*>(o)[0] = w[0];
        reinterpret_cast<uint4*>(o)[1] = w[1];
        return;
      }
    } else if (k0.kind >= 2 && k15.kind == k0.kind && k15.base == k0.base + 15) {
      float* o = e.xbd + k0.base + (size_t)m * d.NS;
      if ((reinterpret_cast<uintptr_t>(o) & 15) == 0) {
        float x[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) x[q] = v[q];
        if (k0.kind == 3) {  // dt columns: softplus with each head's bias
          const int layer = e.layer0 + n0 / e.cols_per_layer;
          const int h0 = (n0 % e.cols_per_layer + e.col_off) - 2 * d.KVD - d.dinner - d.N;
#pragma unroll
          for (int q = 0; q < 16; ++q) x[q] = softplus_f(v[q] + __ldg(&e.dt_bias[layer * d.Hm + h0 + q]));
        } else if (k0.kind == 4) {  // gated-delta writing strength
#pragma unroll
          for (int q = 0; q < 16; ++q) x[q] = sigmoid_f(v[q]);
        }
        float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
        for (int q = 0; q < 4; ++q) o4[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        return;
      }
    }
  }
  for (int j = 0; j < ncols; ++j) ssm_store<__nv_bfloat16>(e, ssm_col(e, n0 + j), m, ro, v[j]);
}

// The committed-row part of the commit epilogue for row m: its ring-row
// offset (-1: not a committed row). n0 is the first column the caller will
// store for the row (column 0 also records the row's position snapshot).
__device__ __forceinline__ long long ssm_kv_row(const Epi& e, int m, int n0) {
  int b;
  long long p;
  epi_row(e, m, b, p, n0);
  return ssm_row_off(e.d, b, p);
}

// Token-major epilogue (swap = 0: output row m = this thread's accumulator
// lane, 16 consecutive output columns n0..n0+15): loads that depend only on
// the row (decay weight of the column's head, segment decay of the row's
// head) are made once per chunk and the state update is vectorised, so the
// epilogue issues no per-element dependent loads.
__device__ __forceinline__ void epi_chunk16(const Epi& e, int m, int n0, int ncols, const float* v) {
  const Dims& d = e.d;
  if (e.kind == EPI_XB && n0 + 16 <= d.dinner && d.P % 16 == 0) {
    const float w = __ldcg(&e.dtw[(size_t)(n0 / d.P) * e.ldt + m]);
    __nv_bfloat16* x = static_cast<__nv_bfloat16*>(e.xsT);
#pragma unroll
    for (int j = 0; j < 16; ++j) x[(size_t)(n0 + j) * e.ldt + m] = __float2bfloat16_rn(w * v[j]);
    return;
  }
  if (e.kind == EPI_STATE && ncols == 16 && d.N % 16 == 0) {
    const float dec = __ldcg(&e.seg_decay[m / d.P]);
    float4* st = reinterpret_cast<float4*>(e.st + (size_t)m * d.N + n0);
    float4 old[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) old[q] = __ldcg(&st[q]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st[q] = make_float4(fmaf(dec, old[q].x, v[4 * q]), fmaf(dec, old[q].y, v[4 * q + 1]),
                          fmaf(dec, old[q].z, v[4 * q + 2]), fmaf(dec, old[q].w, v[4 * q + 3]));
    return;
  }
  if (e.kind == EPI_F32 && ncols == 16 && e.ld % 4 == 0) {  // 16 consecutive outputs of row m
    float4* o = reinterpret_cast<float4*>(e.out + (size_t)m * e.ld + n0);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    return;
  }
  if (e.kind == EPI_RESID && ncols == 16 && e.ld % 8 == 0) {
    const uint4* r = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(e.resid) +
                                                    (size_t)m * e.ld + n0);
    epi_resid16(e, m, n0, v, __ldcg(r), __ldcg(r + 1));
    return;
  }
  if (e.kind == EPI_SSM_KV) {
    epi_ssm_chunk16(e, m, n0, ncols, v, ssm_kv_row(e, m, n0));
    return;
  }
  for (int j = 0; j < ncols; ++j) epi_apply<__nv_bfloat16>(e, m, n0 + j, v[j]);
}

}  // namespace hf
