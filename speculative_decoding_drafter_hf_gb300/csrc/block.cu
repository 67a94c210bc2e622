// Kernels of the full drafter block around the HyFlash layer: the parts a
// real drafter network runs beside the layer's two branches ("HyFlash: A
// Prefix-Memory Prior for On-Device Speculative Decoding" and the
// learnaivisually explainer, "That is HyFlash", describe the two branches of a
// two-layer drafter and name none of these parts; each follows the plainest
// reading of the model families the pages use -- Qwen3 targets, Mamba-2):
//
//   rms_norm      y = x / sqrt(mean(x^2) + 1e-6) * g  (pre-norms, final norm)
//   rope_slots    rotate-half RoPE (base 1e6) of the slot queries and slot
//                 keys at positions pos + s, in place in the fp32 projections
//   gate_skip     y <- (y + D[head] x_s) * silu(z_s) on the memory read
//   swiglu        act = silu(gate) * up
//   argmax_rows   token of a slot = argmax of its logits, ties to the lowest id
//   commit_prep   per committed row: RoPE of the key just appended to the
//                 ring at its position, and Mamba-2's causal depthwise conv1d
//                 (width 4, bias, SiLU) over the row's x | B channels with the
//                 last 3 pre-conv rows carried from earlier commits
//   ring_rope     RoPE of the ring keys a prefill wrote
//   conv_prefill  the same convolution over a prefill pass's tokens, writing
//                 what the chunked scan's x/B step writes (w-scaled x and B,
//                 token-contiguous), and the carried rows after the pass
//
// All of them are small, memory-bound, and launched with programmatic
// dependent launch: each waits for the previous launch before touching data.
#include "common.cuh"

namespace hf {
namespace {

constexpr float kEps = 1e-6f;
constexpr int kConvK = 4;

__device__ __forceinline__ float silu_f(float x) { return x / (1.f + expf(-x)); }

// Rotation of the pair (i, i + dh/2) at position p: cos/sin of p * inv[i],
// inv[i] = theta^(-2i/dh) (a double table made on the host). The angle is
// formed and reduced to [-pi, pi] in double precision -- positions reach 1e5
// and more, where a float angle would be off by ~1e-2 -- then sincosf.
__device__ __forceinline__ void rope_cs(long long p, int i, const double* inv, float* c,
                                        float* s) {
  const double two_pi = 6.283185307179586, inv_two_pi = 0.15915494309189535;
  const double a = (double)p * __ldg(&inv[i]);
  const float r = (float)fma(-rint(a * inv_two_pi), two_pi, a);  // no fp64 division
  sincosf(r, s, c);
}

// ---------------------------------------------------------------- rms_norm
// One CTA per row; fp32 sum of squares.
template <typename T>
__global__ void __launch_bounds__(256) rms_norm_kernel(const T* __restrict__ x,
                                                       const float* __restrict__ g,
                                                       T* __restrict__ y, int D) {
  pdl_wait();
  pdl_trigger();
  const size_t row = blockIdx.x;
  const T* xr = x + row * D;
  float ss = 0.f;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    const float v = to_f(xr[i]);
    ss = fmaf(v, v, ss);
  }
  __shared__ float part[8];
  ss = warp_sum(ss);
  if (threadIdx.x % 32 == 0) part[threadIdx.x / 32] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x / 32); ++w) tot += part[w];
  const float inv = rsqrtf(tot / (float)D + kEps);
  for (int i = threadIdx.x; i < D; i += blockDim.x)
    y[row * D + i] = from_f<T>(to_f(xr[i]) * inv * __ldg(&g[i]));
}

// ---------------------------------------------------------------- rope_slots
// proj rows b*S + s: query heads at [h*dh), slot keys at QD + g*dh; one
// thread per (row, head, pair).
__global__ void rope_slots_kernel(Dims d, int rows, float* __restrict__ proj,
                                  const int64_t* __restrict__ pos,
                                  const double* __restrict__ inv) {
  pdl_wait();
  pdl_trigger();
  const int half = d.dh / 2, heads = d.Hq + d.Hkv;
  const long long total = (long long)rows * heads * half;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(t % half);
    const int hh = (int)((t / half) % heads);
    const int r = (int)(t / ((long long)half * heads));
    const int b = r / d.S, s = r % d.S;
    const long long p = __ldcg(&pos[b]) + s;
    float c, sn;
    rope_cs(p, i, inv, &c, &sn);
    const int col = hh < d.Hq ? hh * d.dh : d.QD + (hh - d.Hq) * d.dh;
    float* v = proj + (size_t)r * d.Nd + col;
    const float lo = v[i], hi = v[i + half];
    v[i] = lo * c - hi * sn;
    v[i + half] = hi * c + lo * sn;
  }
}

// ---------------------------------------------------------------- gate_skip
// mix[r][QD + j] = (y + D[j / P] x_s[j]) * silu(z_s[j]); x_s, z_s at the
// projection columns Nd0 + j and Nd0 + dinner + j (Nd0 = QD + 2 KVD + N).
template <typename T>
__global__ void gate_skip_kernel(Dims d, int rows, T* __restrict__ mix,
                                 const float* __restrict__ proj,
                                 const float* __restrict__ d_skip) {
  pdl_wait();
  pdl_trigger();
  const int nd0 = d.QD + 2 * d.KVD + d.N;
  const long long total = (long long)rows * d.dinner;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(t % d.dinner);
    const int r = (int)(t / d.dinner);
    const float* pr = proj + (size_t)r * d.Nd + nd0;
    T* m = mix + (size_t)r * d.Nz + d.QD + j;
    const float y = to_f(*m) + __ldg(&d_skip[j / d.P]) * pr[j];
    *m = from_f<T>(y * silu_f(pr[d.dinner + j]));
  }
}

// ---------------------------------------------------------------- swiglu
// h [rows][2F] fp32 (gate columns, then up columns) -> act [rows][F].
template <typename T>
__global__ void swiglu_kernel(int rows, int F, const float* __restrict__ h, T* __restrict__ act) {
  pdl_wait();
  pdl_trigger();
  const long long total = (long long)rows * F;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(t % F);
    const size_t r = (size_t)(t / F);
    act[t] = from_f<T>(silu_f(h[r * 2 * F + j]) * h[r * 2 * F + F + j]);
  }
}

// ---------------------------------------------------------------- argmax
// One CTA per row: the largest logit's index, the lowest index among equal
// largest values (NaN never wins).
__global__ void __launch_bounds__(256) argmax_kernel(const float* __restrict__ logits, int V,
                                                     int32_t* __restrict__ tokens) {
  pdl_wait();
  pdl_trigger();
  const size_t row = blockIdx.x;
  const float* lr = logits + row * V;
  float best = -INFINITY;
  int bi = V;  // "none yet": larger than every index
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float v = lr[i];
    if (v > best || (v == best && i < bi)) {
      best = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  __shared__ float sv[8];
  __shared__ int si[8];
  if (threadIdx.x % 32 == 0) {
    sv[threadIdx.x / 32] = best;
    si[threadIdx.x / 32] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x / 32); ++w)
      if (sv[w] > best || (sv[w] == best && si[w] < bi)) {
        best = sv[w];
        bi = si[w];
      }
    tokens[row] = bi < V ? bi : 0;  // all NaN: token 0
  }
}

// ---------------------------------------------------------------- commit_prep
// Grid (ceil((C + Hkv*dh/2) / 256), B, L), C = dinner + N. Thread index
// u < C: conv channel u of (layer, request); else RoPE pair u - C of the keys
// the commit projection appended for the accepted rows. Counts outside
// 0..S+1 are treated as 0 (the state kernel flags them).
template <typename T>
__global__ void commit_prep_kernel(Dims d, const int32_t* __restrict__ n_acc,
                                   const int64_t* __restrict__ pos, T* __restrict__ ring_k,
                                   float* __restrict__ xbd, long long xls,
                                   float* __restrict__ conv_state, const float* __restrict__ conv_w,
                                   const float* __restrict__ conv_b,
                                   const double* __restrict__ inv) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y, l = blockIdx.z;
  const int lim = d.S + 1;
  const int nr = __ldcg(&n_acc[b]);
  const int n = (nr >= 0 && nr <= lim) ? nr : 0;
  if (n == 0) return;
  const int C = d.dinner + d.N;
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  const long long p0 = __ldcg(&pos[b]);
  if (u < C) {
    float* xb = xbd + (size_t)l * xls + (size_t)b * lim * d.NS + u;
    float* cs = conv_state + (((size_t)l * d.Bmax + b) * (kConvK - 1)) * C + u;
    const float* w = conv_w + ((size_t)l * C + u) * kConvK;
    const float bias = __ldg(&conv_b[(size_t)l * C + u]);
    // rolling window of the last 3 pre-conv rows (h0 oldest), in registers
    float h0 = cs[0], h1 = cs[(size_t)C], h2 = cs[(size_t)2 * C];
    const float w0 = __ldg(&w[0]), w1 = __ldg(&w[1]), w2 = __ldg(&w[2]), w3 = __ldg(&w[3]);
    for (int t = 0; t < n; ++t) {
      const float x = xb[(size_t)t * d.NS];
      xb[(size_t)t * d.NS] = silu_f(fmaf(w3, x, fmaf(w2, h2, fmaf(w1, h1, fmaf(w0, h0, bias)))));
      h0 = h1;
      h1 = h2;
      h2 = x;
    }
    cs[0] = h0;
    cs[(size_t)C] = h1;
    cs[(size_t)2 * C] = h2;
    return;
  }
  const int half = d.dh / 2;
  const int q = u - C;
  if (q >= d.Hkv * half) return;
  const int g = q / half, i = q % half;
  T* base = ring_k + (((size_t)l * d.Bmax + b) * d.Hkv + g) * d.W * d.dh;
  for (int t = 0; t < n; ++t) {
    const long long p = p0 + t;
    float c, s;
    rope_cs(p, i, inv, &c, &s);
    T* v = base + (size_t)(p % d.W) * d.dh;
    const float lo = to_f(v[i]), hi = to_f(v[i + half]);
    v[i] = from_f<T>(lo * c - hi * s);
    v[i + half] = from_f<T>(hi * c + lo * s);
  }
}

// ---------------------------------------------------------------- ring_rope
// Prefill window rows r (request row_req[r], position row_pos[r]) of one
// layer: RoPE of the keys the window GEMM wrote.
template <typename T>
__global__ void ring_rope_kernel(Dims d, int layer, int rows, const int32_t* __restrict__ row_req,
                                 const int64_t* __restrict__ row_pos, T* __restrict__ ring_k,
                                 const double* __restrict__ inv) {
  pdl_wait();
  pdl_trigger();
  const int half = d.dh / 2;
  const long long total = (long long)rows * d.Hkv * half;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(t % half);
    const int g = (int)((t / half) % d.Hkv);
    const int r = (int)(t / ((long long)half * d.Hkv));
    const int b = __ldcg(&row_req[r]);
    const long long p = __ldcg(&row_pos[r]);
    float c, s;
    rope_cs(p, i, inv, &c, &s);
    T* v = ring_k + ((((size_t)layer * d.Bmax + b) * d.Hkv + g) * d.W + p % d.W) * d.dh;
    const float lo = to_f(v[i]), hi = to_f(v[i + half]);
    v[i] = from_f<T>(lo * c - hi * s);
    v[i + half] = from_f<T>(hi * c + lo * s);
  }
}

// ---------------------------------------------------------------- conv_prefill
// Pass of T tokens of one (layer, request). U [T][C] fp32: pre-conv x | B
// rows; hist [3][C]: the 3 pre-conv rows before the pass. Tile of 32
// channels x 32 tokens per CTA (32 x 8 threads): the 35 rows it needs are
// staged in shared memory (reads along channels), outputs written along
// tokens: x channels to xsT[c][t] = w[c / P][t] * silu(conv), B channels to
// bT[c - dinner][t] = silu(conv), both token-contiguous with row length ldt.
template <typename T>
__global__ void __launch_bounds__(256) conv_prefill_kernel(
    Dims d, int Tn, int ldt, const float* __restrict__ U, const float* __restrict__ hist,
    const float* __restrict__ dtw, const float* __restrict__ conv_w,
    const float* __restrict__ conv_b, T* __restrict__ xsT, T* __restrict__ bT) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[32 + kConvK - 1][33];
  const int C = d.dinner + d.N;
  const int c0 = blockIdx.x * 32, t0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int rr = ty; rr < 32 + kConvK - 1; rr += 8) {
    const int t = t0 + rr - (kConvK - 1);  // token of staged row rr
    const int c = c0 + tx;
    float v = 0.f;
    if (c < C && t < Tn) v = t >= 0 ? U[(size_t)t * C + c] : hist[(size_t)(t + kConvK - 1) * C + c];
    tile[rr][tx] = v;
  }
  __syncthreads();
  // thread (tx, ty): token t0 + tx, channels c0 + ty + 8 k
  const int t = t0 + tx;
  if (t >= Tn) return;
  for (int k = 0; k < 4; ++k) {
    const int cl = ty + 8 * k, c = c0 + cl;
    if (c >= C) break;
    const float* w = conv_w + (size_t)c * kConvK;
    float acc = __ldg(&conv_b[c]);
#pragma unroll
    for (int j = 0; j < kConvK; ++j) acc = fmaf(__ldg(&w[j]), tile[tx + j][cl], acc);
    const float u = silu_f(acc);
    if (c < d.dinner)
      xsT[(size_t)c * ldt + t] = from_f<T>(__ldcg(&dtw[(size_t)(c / d.P) * ldt + t]) * u);
    else
      bT[(size_t)(c - d.dinner) * ldt + t] = from_f<T>(u);
  }
}

// The carried rows after a pass: hist[k] <- (T + k < 3) ? hist[T + k] : U[T + k - 3].
__global__ void conv_carry_kernel(int C, int Tn, const float* __restrict__ U,
                                  float* __restrict__ hist) {
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  float nv[kConvK - 1];
  for (int k = 0; k < kConvK - 1; ++k)
    nv[k] = Tn + k < kConvK - 1 ? hist[(size_t)(Tn + k) * C + c]
                                : U[(size_t)(Tn + k - (kConvK - 1)) * C + c];
  for (int k = 0; k < kConvK - 1; ++k) hist[(size_t)k * C + c] = nv[k];
}

// Zero the carried rows of the named requests (all layers) before a prefill.
__global__ void conv_reset_kernel(Dims d, int n_req, const int32_t* __restrict__ reqs,
                                  float* __restrict__ conv_state) {
  pdl_wait();
  pdl_trigger();
  const int C = d.dinner + d.N;
  const long long per = (long long)(kConvK - 1) * C;
  const long long total = (long long)d.L * n_req * per;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long e = t % per;
    const int i = (int)((t / per) % n_req);
    const int l = (int)(t / (per * n_req));
    conv_state[((size_t)l * d.Bmax + __ldcg(&reqs[i])) * per + e] = 0.f;
  }
}

int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 8 * 152) g = 8 * 152;
  return (int)g;
}

}  // namespace

cudaError_t launch_rms_norm(int dtype, const void* x, const float* g, void* y, int rows, int D,
                            cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == HF_F32)
    return launch_pdl(rms_norm_kernel<float>, dim3(rows), dim3(256), 0, st,
                      static_cast<const float*>(x), g, static_cast<float*>(y), D);
  return launch_pdl(rms_norm_kernel<__nv_bfloat16>, dim3(rows), dim3(256), 0, st,
                    static_cast<const __nv_bfloat16*>(x), g, static_cast<__nv_bfloat16*>(y), D);
}

cudaError_t launch_rope_slots(const Dims& d, int rows, float* proj, const int64_t* pos,
                              const double* inv, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const long long work = (long long)rows * (d.Hq + d.Hkv) * (d.dh / 2);
  return launch_pdl(rope_slots_kernel, dim3(grid_for(work, 256)), dim3(256), 0, st, d, rows, proj,
                    pos, inv);
}

cudaError_t launch_gate_skip(int dtype, const Dims& d, int rows, void* mix, const float* proj,
                             const float* d_skip, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid(grid_for((long long)rows * d.dinner, 256));
  if (dtype == HF_F32)
    return launch_pdl(gate_skip_kernel<float>, grid, dim3(256), 0, st, d, rows,
                      static_cast<float*>(mix), proj, d_skip);
  return launch_pdl(gate_skip_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, d, rows,
                    static_cast<__nv_bfloat16*>(mix), proj, d_skip);
}

cudaError_t launch_swiglu(int dtype, int rows, int F, const float* h, void* act, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid(grid_for((long long)rows * F, 256));
  if (dtype == HF_F32)
    return launch_pdl(swiglu_kernel<float>, grid, dim3(256), 0, st, rows, F, h,
                      static_cast<float*>(act));
  return launch_pdl(swiglu_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, rows, F, h,
                    static_cast<__nv_bfloat16*>(act));
}

cudaError_t launch_argmax(int rows, int V, const float* logits, int32_t* tokens, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(argmax_kernel, dim3(rows), dim3(256), 0, st, logits, V, tokens);
}

cudaError_t launch_commit_prep(int dtype, const Dims& d, int B, const int32_t* n_acc,
                               const int64_t* pos, void* ring_k, float* xbd, long long xls,
                               float* conv_state, const float* conv_w, const float* conv_b,
                               const double* inv, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  if (d.S + 1 > 17) return cudaErrorInvalidValue;
  const int work = d.dinner + d.N + d.Hkv * (d.dh / 2);
  const dim3 grid((work + 255) / 256, B, d.L);
  if (dtype == HF_F32)
    return launch_pdl(commit_prep_kernel<float>, grid, dim3(256), 0, st, d, n_acc, pos,
                      static_cast<float*>(ring_k), xbd, xls, conv_state, conv_w, conv_b, inv);
  return launch_pdl(commit_prep_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, d, n_acc, pos,
                    static_cast<__nv_bfloat16*>(ring_k), xbd, xls, conv_state, conv_w, conv_b, inv);
}

cudaError_t launch_ring_rope(int dtype, const Dims& d, int layer, int rows, const int32_t* row_req,
                             const int64_t* row_pos, void* ring_k, const double* inv,
                             cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid(grid_for((long long)rows * d.Hkv * (d.dh / 2), 256));
  if (dtype == HF_F32)
    return launch_pdl(ring_rope_kernel<float>, grid, dim3(256), 0, st, d, layer, rows, row_req,
                      row_pos, static_cast<float*>(ring_k), inv);
  return launch_pdl(ring_rope_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, d, layer, rows,
                    row_req, row_pos, static_cast<__nv_bfloat16*>(ring_k), inv);
}

cudaError_t launch_conv_prefill(int dtype, const Dims& d, int Tn, int ldt, const float* U,
                                float* hist, const float* dtw, const float* conv_w,
                                const float* conv_b, void* xsT, void* bT, cudaStream_t st) {
  if (Tn <= 0) return cudaSuccess;
  const int C = d.dinner + d.N;
  const dim3 grid((C + 31) / 32, (Tn + 31) / 32), blk(32, 8);
  cudaError_t e;
  if (dtype == HF_F32)
    e = launch_pdl(conv_prefill_kernel<float>, grid, blk, 0, st, d, Tn, ldt, U,
                   static_cast<const float*>(hist), dtw, conv_w, conv_b, static_cast<float*>(xsT),
                   static_cast<float*>(bT));
  else
    e = launch_pdl(conv_prefill_kernel<__nv_bfloat16>, grid, blk, 0, st, d, Tn, ldt, U,
                   static_cast<const float*>(hist), dtw, conv_w, conv_b,
                   static_cast<__nv_bfloat16*>(xsT), static_cast<__nv_bfloat16*>(bT));
  if (e != cudaSuccess) return e;
  return launch_pdl(conv_carry_kernel, dim3((C + 255) / 256), dim3(256), 0, st, C, Tn, U, hist);
}

cudaError_t launch_conv_reset(const Dims& d, int n_req, const int32_t* reqs, float* conv_state,
                              cudaStream_t st) {
  if (n_req <= 0) return cudaSuccess;
  const long long work = (long long)d.L * n_req * 3 * (d.dinner + d.N);
  return launch_pdl(conv_reset_kernel, dim3(grid_for(work, 256)), dim3(256), 0, st, d, n_req, reqs,
                    conv_state);
}

}  // namespace hf
