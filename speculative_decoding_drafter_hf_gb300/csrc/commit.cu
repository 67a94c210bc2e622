// Commit path: the sequential memory update, with the accepted-count check,
// the packed offsets, the ring tags and the position update.
//
// Source: learnaivisually explainer, FAQ "Why does the memory update only
// from committed features?" and "That is HyFlash": after verification only
// the newly committed features update the state, in order; drafting never
// writes it. Ring slots follow the sliding-window rule (Jargon,
// "Sliding-window attention"): the window keeps the most recent W committed
// positions, position t in slot t mod W. The K/V ring append itself happens
// in the commit projection's epilogue (common.cuh, EPI_SSM_KV).
#include <mutex>

#include "common.cuh"

namespace hf {
namespace {

constexpr int THREADS_CS = 256;
constexpr int QPT_HEAD = 8;  // float4 elements per thread when one CTA holds a whole head (P*N <= 8192)

// Shared memory of the state-update kernel: staged x / B / dt rows (and C
// when the memory read is fused), then the padded copy of the new state and
// the k-part sums of the memory read.
struct CsLayout {
  size_t sx, sb, sd, sbeta, sxo, sbo, sdo, wsum, rows, red, qn, total;  // float offsets
};
__host__ __device__ inline CsLayout cs_layout(const Dims& d, bool read) {
  CsLayout m{};
  const int lim = d.S + 1;
  m.sx = 0;
  m.sb = m.sx + (size_t)lim * d.P;
  m.sd = m.sb + (size_t)lim * d.N;
  m.sbeta = m.sd + ((lim + 3) & ~3);  // gated delta: writing strengths
  m.sxo = m.sbeta + (d.gdn ? (size_t)((lim + 3) & ~3) : 0);
  // memory horizon M > 1: the rows leaving the horizon, and a reduction slot
  m.sbo = m.sxo + (d.Mr > 0 ? (size_t)lim * d.P : 0);
  m.sdo = m.sbo + (d.Mr > 0 ? (size_t)lim * d.N : 0);
  m.wsum = m.sdo + (d.Mr > 0 ? (size_t)((lim + 3) & ~3) : 0);
  m.rows = m.wsum + (d.Mr > 0 ? 32 : 0);
  m.red = m.rows + (read ? (size_t)d.P * (d.N + 8) : 0);
  m.qn = m.red + (read ? (size_t)mem_ksplit(d) * d.P * 8 : 0);
  m.total = m.qn + (read ? 16 : 0);  // gated delta: 1/|C_s| of the slots
  return m;
}

// One gated-delta row applied to a thread's QPT float4 of a head's state
// (state rows of gsz consecutive lanes; k4: this lane's 4 columns of B, not
// yet normalised): S <- al (S - be (S k) k^T) + be x k^T, k = B/|B|, written
// as S <- al S + be (x - al (S k)) k^T.
template <int QPT>
__device__ __forceinline__ void gdn_token(float4 (&hv)[QPT], const float (&xv)[QPT], float4 k4,
                                          float al, float be, int gsz) {
  float ss = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
  for (int o = 1; o < gsz; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float kn = 1.f / sqrtf(ss);
  k4 = make_float4(k4.x * kn, k4.y * kn, k4.z * kn, k4.w * kn);
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    float dot = hv[u].x * k4.x + hv[u].y * k4.y + hv[u].z * k4.z + hv[u].w * k4.w;
    for (int o = 1; o < gsz; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float cf = be * (xv[u] - al * dot);
    hv[u].x = fmaf(al, hv[u].x, cf * k4.x);
    hv[u].y = fmaf(al, hv[u].y, cf * k4.y);
    hv[u].z = fmaf(al, hv[u].z, cf * k4.z);
    hv[u].w = fmaf(al, hv[u].w, cf * k4.w);
  }
}

constexpr int QPT_SCAN = 2;

// Gated-delta prefill of one request and layer over T tokens, whose x | B |
// dt | beta rows (stride NS) the projection left in xs: grid (Hm * qsplit),
// CTA (h * qsplit + q) keeps its slice of head h's state in registers and
// applies the tokens in order; the next token's inputs are loaded while the
// current one is applied.
__global__ void __launch_bounds__(THREADS_CS)
gdn_prefill_kernel(Dims d, int l, int b, int T, int qsplit, const float* __restrict__ xs,
                   const float* __restrict__ A_log, float* __restrict__ state) {
  const int hd = blockIdx.x / qsplit, qs = blockIdx.x % qsplit;
  const int P = d.P, N = d.N, nq = P * N / 4;
  float4* h = reinterpret_cast<float4*>(state + ((((size_t)l * d.Bmax + b) * d.Hm + hd) * P) * N);
  const int q0 = qs * QPT_SCAN * THREADS_CS;
  float4 hv[QPT_SCAN];
  int pi[QPT_SCAN];
  int ci = 0;
#pragma unroll
  for (int u = 0; u < QPT_SCAN; ++u) {  // elements past the head: index 0, never stored
    const int q = q0 + threadIdx.x + u * THREADS_CS;
    const bool in = q < nq;
    hv[u] = in ? __ldcg(&h[q]) : make_float4(0.f, 0.f, 0.f, 0.f);
    pi[u] = in ? (q * 4) / N : 0;
    if (u == 0) ci = in ? (q * 4) % N : 0;
  }
  const float A = -expf(__ldg(&A_log[l * d.Hm + hd]));
  const int gsz = N / 4;
  const size_t cx = (size_t)hd * P, cb = d.dinner, cd = (size_t)d.dinner + N + hd,
               cbe = (size_t)d.dinner + N + d.Hm + hd;
  float xv[QPT_SCAN], dt = 0.f, be = 0.f;
  float4 kb = make_float4(0.f, 0.f, 0.f, 0.f);
  if (T > 0) {
#pragma unroll
    for (int u = 0; u < QPT_SCAN; ++u) xv[u] = __ldcg(&xs[cx + pi[u]]);
    kb = __ldcg(reinterpret_cast<const float4*>(xs + cb + ci));
    dt = __ldcg(&xs[cd]);
    be = __ldcg(&xs[cbe]);
  }
  for (int t = 0; t < T; ++t) {
    float xn[QPT_SCAN], dn = 0.f, bn = 0.f;
    float4 kn = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t + 1 < T) {
      const float* row = xs + (size_t)(t + 1) * d.NS;
#pragma unroll
      for (int u = 0; u < QPT_SCAN; ++u) xn[u] = __ldcg(&row[cx + pi[u]]);
      kn = __ldcg(reinterpret_cast<const float4*>(row + cb + ci));
      dn = __ldcg(&row[cd]);
      bn = __ldcg(&row[cbe]);
    }
    gdn_token<QPT_SCAN>(hv, xv, kb, expf(dt * A), be, gsz);
#pragma unroll
    for (int u = 0; u < QPT_SCAN; ++u) xv[u] = xn[u];
    kb = kn;
    dt = dn;
    be = bn;
  }
#pragma unroll
  for (int u = 0; u < QPT_SCAN; ++u) {
    const int q = q0 + threadIdx.x + u * THREADS_CS;
    if (q < nq) h[q] = hv[u];
  }
}

// grid (Hm * qsplit, B, L): CTA (h * qsplit + q, b, l) takes the q-th of
// qsplit slices (QPT float4 per thread, whole state rows) of the state of
// one (layer, request, head), reads it once (all loads in flight together),
// advances it over the request's accepted rows in order, and writes it once.
// Small batches split a head over several CTAs (more loads in flight);
// large batches, and the fused memory read, take a whole head per CTA.
// CTA (0, b, 0) also checks n_b, writes offsets[b] (and offsets[B]), the
// ring tags of the appended positions, and pos[b] += n_b.
//
// early: the previous launch signalled its dependents after its own wait, so
// the state, positions and counts are final at launch: they are read before
// this launch's wait (only the staged projections come from that launch).
// late: signal dependents only after this launch's own wait, so that the
// next launch may read what the launches before this one wrote.
//
// With memC set, the layer-0 CTAs also make the next draft's memory read on
// the state they hold, once it is final: y[s, p] = sum_n h[p, n] C[s, n]
// (C: the slot projections of that draft, rows b*S + s with stride Nd) on
// the tensor cores from a padded shared-memory copy of the new state, into
// mix[b*S + s][QD + h*P + p] -- the values the draft-time read would
// produce, without reading the state a second time.
//
// Memory horizon M (the paper's "SSM: Last feature" / "SSM: Last 512"
// interventions: the memory is the fold, from zero, of the last M committed
// features). M = 1: the new state is the last accepted row's term alone (the
// old state is not read). M > 1: each accepted row at position p adds its
// term and removes the term of the feature at position q = p - M, which
// leaves the horizon; in the state after p that feature's weight is
// dt_q * exp(A * sum_{s=q+1..p} dt_s), so
//   h <- exp(dt_p A) h + dt_p x_p B_p^T - dt_q exp(A W_p) x_q B_q^T,
//   W_p = sum of dt over positions q+1..p.
// x, B and dt of the last Mr = M + S + 1 committed features sit in a ring
// (row = position mod Mr); a commit reads rows of positions < T (its first
// position, recorded by the commit projection) and writes rows T..T+n-1,
// never the same rows (n <= S + 1). W is recomputed from the ring every
// commit, so no running sum drifts.
//
// Gated-delta memory (gdn_token; MODE 2): per accepted row, with the unit
// key k = B/|B| (|B| summed over the lanes that hold one state row),
// alpha = exp(dt A) and beta the row's writing strength,
//   S <- alpha (S - beta (S k) k^T) + beta x k^T,
// where (S k) of a state row is a sum over the lanes holding that row.
// MODE: 0 Mamba-2, 1 Mamba-2 with a horizon ring (M > 1), 2 gated delta.
template <typename T, int QPT, int MODE>
__global__ void __launch_bounds__(THREADS_CS)
commit_state_kernel(Dims d, int B, int qsplit, int early, int late,
                    const int32_t* __restrict__ n_acc,
                    const float* __restrict__ xbd, long long xls,
                    const float* __restrict__ A_log, float* __restrict__ state,
                    int64_t* __restrict__ pos, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ tags, int32_t* __restrict__ err,
                    const float* __restrict__ memC, T* __restrict__ mix, MemRing mr) {
  extern __shared__ __align__(16) float sm[];
  if (!late) pdl_trigger();
  if (!early) {
    pdl_wait();
    if (late) pdl_trigger();
  }
  const int hd = blockIdx.x / qsplit, qs = blockIdx.x % qsplit, b = blockIdx.y, l = blockIdx.z;
  const int lim = d.S + 1;
  const int n_raw = __ldcg(&n_acc[b]);
  const bool valid = n_raw >= 0 && n_raw <= lim;
  const int n = valid ? n_raw : 0;
  const bool read = memC != nullptr && l == 0;  // (then qsplit == 1)
  const bool bookkeeper = blockIdx.x == 0 && l == 0;
  if (n == 0 && !read && !bookkeeper) return;
  const int P = d.P, N = d.N;
  float4* h = reinterpret_cast<float4*>(state + ((((size_t)l * d.Bmax + b) * d.Hm + hd) * P) * N);
  const int nq = P * N / 4;
  const int q0 = qs * QPT * THREADS_CS;
  const bool work = n > 0 || read;
  const bool last_only = d.Mh == 1;       // memory = the last accepted row's term
  const bool fresh = last_only && n > 0;  // (then the old state is not needed)
  float4 hv[QPT];
  int pi[QPT], ci[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {  // elements past the head: index 0 (in bounds), never stored
    const int q = q0 + threadIdx.x + u * THREADS_CS;
    const bool in = work && q < nq;
    hv[u] = in && !fresh ? __ldcg(&h[q]) : make_float4(0.f, 0.f, 0.f, 0.f);
    pi[u] = in ? (q * 4) / N : 0;
    ci[u] = in ? (q * 4) % N : 0;
  }
  // The previous launch (the commit projection) reads the positions in its
  // epilogue and writes the staged rows: wait before touching either.
  if (early) {
    pdl_wait();
    if (late) pdl_trigger();
  }
  if (bookkeeper) {
    __shared__ long long s_pos;
    if (threadIdx.x < 32) {
      int part = 0;
      for (int i = threadIdx.x; i < b; i += 32) {
        const int m = __ldcg(&n_acc[i]);
        part += (m >= 0 && m <= lim) ? m : 0;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (threadIdx.x == 0) {
        if (!valid) atomicOr(err, ERR_BAD_ACCEPTED);
        offsets[b] = part;
        if (b == B - 1) offsets[B] = part + n;
        s_pos = __ldcg(&pos[b]);
      }
    }
    __syncthreads();
    const long long p0 = s_pos;
    for (int t = threadIdx.x; t < n; t += blockDim.x)
      tags[(size_t)b * d.W + (int)((p0 + t) % d.W)] = (int32_t)(p0 + t);
    if (threadIdx.x == 0) pos[b] = p0 + n;
  }
  if (!work) return;
  // stage x (this head), B and dt of the n accepted rows b*(S+1) + t
  const CsLayout L = cs_layout(d, read);
  float* sx = sm + L.sx;  // [lim][P]
  float* sb = sm + L.sb;  // [lim][N]
  float* sd = sm + L.sd;  // [lim]
  const float* xb = xbd + (size_t)l * xls + (size_t)b * lim * d.NS;
  for (int i = threadIdx.x; i < n * (P / 4); i += blockDim.x) {
    const int t = i / (P / 4), c = (i % (P / 4)) * 4;
    *reinterpret_cast<float4*>(&sx[t * P + c]) =
        __ldcg(reinterpret_cast<const float4*>(xb + (size_t)t * d.NS + hd * P + c));
  }
  for (int i = threadIdx.x; i < n * (N / 4); i += blockDim.x) {
    const int t = i / (N / 4), c = (i % (N / 4)) * 4;
    *reinterpret_cast<float4*>(&sb[t * N + c]) =
        __ldcg(reinterpret_cast<const float4*>(xb + (size_t)t * d.NS + d.dinner + c));
  }
  for (int t = threadIdx.x; t < n; t += blockDim.x)
    sd[t] = __ldcg(&xb[(size_t)t * d.NS + d.dinner + N + hd]);
  __syncthreads();
  const float A = -expf(__ldg(&A_log[l * d.Hm + hd]));
  const bool ring = MODE == 1 && n > 0;
  constexpr bool GDN = MODE == 2;
  float* sbeta = sm + L.sbeta;
  if (GDN) {
    for (int t = threadIdx.x; t < n; t += blockDim.x)
      sbeta[t] = __ldcg(&xb[(size_t)t * d.NS + d.dinner + N + d.Hm + hd]);
    __syncthreads();
  }
  float* sxo = sm + L.sxo;  // [lim][P]: x of the rows leaving the horizon (0: none)
  float* sbo = sm + L.sbo;  // [lim][N]
  float* sdo = sm + L.sdo;  // [lim]
  float wbase = 0.f;        // sum of dt over positions T - M .. T - 1
  if (ring) {
    const long long T0 = __ldcg(&mr.pos_snap[b]);
    const int Mh = d.Mh, Mr = d.Mr;
    const int r0 = (int)(T0 % Mr);  // ring row of position T0 (one 64-bit modulo)
    // ring row of position T0 + k, -Mr <= k < Mr
    auto row_of = [&](int k) { int r = r0 + k; r += r < 0 ? Mr : 0; return r >= Mr ? r - Mr : r; };
    const size_t lb = (size_t)l * d.Bmax + b;
    const float* dtr = mr.dt + (lb * d.Hm + hd) * Mr;
    const int cnt = (int)(T0 < Mh ? T0 : Mh);  // positions T0 - cnt .. T0 - 1 in the horizon
    float part = 0.f;
    for (int k = (int)threadIdx.x; k < cnt; k += blockDim.x) part += __ldcg(&dtr[row_of(k - cnt)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    float* wsum = sm + L.wsum;
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = part;
    // leaving rows: position q = T + t - M; older than the commit -> ring,
    // inside it (M <= S) -> staged rows; negative -> no row
    for (int i = threadIdx.x; i < n * (P / 4); i += blockDim.x) {
      const int t = i / (P / 4), c = (i % (P / 4)) * 4;
      const long long q = T0 + t - Mh;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q >= T0)
        v = *reinterpret_cast<const float4*>(&sx[(int)(q - T0) * P + c]);
      else if (q >= 0)
        v = __ldcg(reinterpret_cast<const float4*>(mr.x + (lb * Mr + row_of(t - Mh)) * d.dinner + hd * P + c));
      *reinterpret_cast<float4*>(&sxo[t * P + c]) = v;
    }
    for (int i = threadIdx.x; i < n * (N / 4); i += blockDim.x) {
      const int t = i / (N / 4), c = (i % (N / 4)) * 4;
      const long long q = T0 + t - Mh;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q >= T0)
        v = *reinterpret_cast<const float4*>(&sb[(int)(q - T0) * N + c]);
      else if (q >= 0)
        v = __ldcg(reinterpret_cast<const float4*>(mr.b + (lb * Mr + row_of(t - Mh)) * N + c));
      *reinterpret_cast<float4*>(&sbo[t * N + c]) = v;
    }
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
      const long long q = T0 + t - Mh;
      sdo[t] = q >= T0 ? sd[(int)(q - T0)] : (q >= 0 ? __ldcg(&dtr[row_of(t - Mh)]) : 0.f);
    }
    // the new rows into the ring (one CTA per head; head 0 also writes B)
    if (qs == 0) {
      for (int i = threadIdx.x; i < n * (P / 4); i += blockDim.x) {
        const int t = i / (P / 4), c = (i % (P / 4)) * 4;
        *reinterpret_cast<float4*>(mr.x + (lb * Mr + row_of(t)) * d.dinner + hd * P + c) =
            *reinterpret_cast<const float4*>(&sx[t * P + c]);
      }
      for (int t = threadIdx.x; t < n; t += blockDim.x)
        mr.dt[(lb * d.Hm + hd) * Mr + row_of(t)] = sd[t];
      if (hd == 0)
        for (int i = threadIdx.x; i < n * (N / 4); i += blockDim.x) {
          const int t = i / (N / 4), c = (i % (N / 4)) * 4;
          *reinterpret_cast<float4*>(mr.b + (lb * Mr + row_of(t)) * N + c) =
              *reinterpret_cast<const float4*>(&sb[t * N + c]);
        }
    }
    __syncthreads();
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) wbase += wsum[w];
  }
  float W = wbase;  // sum of dt over the horizon ending at the current row
  if (GDN) {
    const int gsz = N / 4;  // lanes holding one state row
    for (int t = 0; t < n; ++t) {
      float xv[QPT];
#pragma unroll
      for (int u = 0; u < QPT; ++u) xv[u] = sx[t * P + pi[u]];
      gdn_token<QPT>(hv, xv, *reinterpret_cast<const float4*>(&sb[t * N + ci[0]]),
                     expf(sd[t] * A), sbeta[t], gsz);
    }
  }
  for (int t = 0; t < (GDN ? 0 : n); ++t) {
    const float dt = sd[t];
    const float dec = last_only ? 0.f : expf(dt * A);
    float co = 0.f;  // weight of the row leaving the horizon
    if (ring) {
      W += dt - sdo[t];
      co = sdo[t] * expf(A * W);
    }
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const float xv = dt * sx[t * P + pi[u]];
      const float4 Bv = *reinterpret_cast<const float4*>(&sb[t * N + ci[u]]);
      hv[u].x = fmaf(dec, hv[u].x, xv * Bv.x);
      hv[u].y = fmaf(dec, hv[u].y, xv * Bv.y);
      hv[u].z = fmaf(dec, hv[u].z, xv * Bv.z);
      hv[u].w = fmaf(dec, hv[u].w, xv * Bv.w);
      if (ring) {
        const float xo = co * sxo[t * P + pi[u]];
        const float4 Bo = *reinterpret_cast<const float4*>(&sbo[t * N + ci[u]]);
        hv[u].x = fmaf(-xo, Bo.x, hv[u].x);
        hv[u].y = fmaf(-xo, Bo.y, hv[u].y);
        hv[u].z = fmaf(-xo, Bo.z, hv[u].z);
        hv[u].w = fmaf(-xo, Bo.w, hv[u].w);
      }
    }
  }
  if (n > 0) {
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int q = q0 + threadIdx.x + u * THREADS_CS;
      if (q < nq) h[q] = hv[u];
    }
  }
  if (!read) return;

  // ---- memory read of the new state (tensor cores; see common.cuh)
  const int RS = N + 8;  // padded row stride (floats): A-fragment loads conflict-free
  float* rows = sm + L.rows;
  float* red = sm + L.red;
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int q = q0 + threadIdx.x + u * THREADS_CS;
    if (q < nq) *reinterpret_cast<float4*>(&rows[pi[u] * RS + ci[u]]) = hv[u];
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int MT = P / 16, KSPL = mem_ksplit(d), G16 = N / 16 / KSPL;
  const int mt = warp % MT, kp = warp / MT;
  const bool active = kp < KSPL;
  const int r0 = mt * 16 + g8;
  const int col0 = kp * G16 * 16 + 4 * t4;
  uint32_t bf[MEM_G16][4];
  {
    const float* crow = memC + ((size_t)b * d.S + g8) * d.Nd + col0;
#pragma unroll
    for (int j = 0; j < MEM_G16; ++j) {
      float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && j < G16 && g8 < d.S) c = __ldcg(reinterpret_cast<const float4*>(crow + j * 16));
      bf[j][0] = to_tf32(c.x);
      bf[j][1] = to_tf32(c.y);
      bf[j][2] = to_tf32(c.z);
      bf[j][3] = to_tf32(c.w);
    }
  }
  float* qn = sm + L.qn;
  if (GDN) {  // read with q = C_s / |C_s|
    const int nw = blockDim.x >> 5;
    for (int s2 = warp; s2 < d.S; s2 += nw) {
      float acc = 0.f;
      for (int c = lane; c < N; c += 32) {
        const float v = __ldcg(&memC[((size_t)b * d.S + s2) * d.Nd + c]);
        acc = fmaf(v, v, acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) qn[s2] = 1.f / sqrtf(acc);
    }
  }
  __syncthreads();  // the new state is in shared memory
  if (active) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < MEM_G16; ++j)
      if (j < G16) {
        const float4 x0 = *reinterpret_cast<const float4*>(&rows[r0 * RS + col0 + j * 16]);
        const float4 x1 = *reinterpret_cast<const float4*>(&rows[(r0 + 8) * RS + col0 + j * 16]);
        mma_tf32_1688(c, to_tf32(x0.x), to_tf32(x1.x), to_tf32(x0.y), to_tf32(x1.y), bf[j][0],
                      bf[j][1]);
        mma_tf32_1688(c, to_tf32(x0.z), to_tf32(x1.z), to_tf32(x0.w), to_tf32(x1.w), bf[j][2],
                      bf[j][3]);
      }
    float* rp = red + ((size_t)kp * P + r0) * 8 + 2 * t4;
    *reinterpret_cast<float2*>(rp) = make_float2(c[0], c[1]);
    *reinterpret_cast<float2*>(rp + 64) = make_float2(c[2], c[3]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < d.S * P; e += blockDim.x) {
    const int sl = e / P, p = e % P;
    float y = 0.f;
    for (int q = 0; q < KSPL; ++q) y += red[((size_t)q * P + p) * 8 + sl];
    if (GDN) y *= qn[sl];
    mix[((size_t)b * d.S + sl) * d.Nz + d.QD + (size_t)hd * P + p] = from_f<T>(y);
  }
}


// ---------------------------------------------------------------------------
// Pipelined state update for large batches (Mamba-2 memory without a
// horizon). The per-head kernel above loads a head, updates it and stores it
// with nothing else in flight, so at 64 requests the SMs wait on load latency
// (three CTAs per SM, ~3.5 TB/s). Here a persistent grid of one CTA per SM
// walks the (layer, request, head) items i = blockIdx.x + k * gridDim.x,
// warp-specialised:
//   producer warp: per item, one bulk copy of the head's state (P*N fp32)
//     into a shared-memory stage, and 16-byte async copies of the accepted
//     rows' x, B (and for a layer-0 read the draft's C rows), dt and A_log,
//     all completing on the stage's "full" barrier; PIPE_ST stages ahead;
//   16 consumer warps: wait on "full", fold the rows into the state in
//     registers in order (the update of the per-head kernel), store the
//     new state, and release the stage on its "empty" barrier. Layer-0
//     items also make the next draft's memory read when memC is set (the
//     consumers synchronise among themselves only there).
// Items with n = 0 and no read are skipped; the producer warp also does the
// bookkeeping (count check, offsets, tags, pos) of the requests whose
// (layer 0, head 0) item its CTA owns.
constexpr int PIPE_CWARPS = 16;                  // consumer warps
constexpr int PIPE_CT = PIPE_CWARPS * 32;        // consumer threads
constexpr int PIPE_THREADS = PIPE_CT + 32;       // + the producer warp
constexpr int PIPE_QPT = 4;    // float4 of the state per consumer thread (P*N <= 8192)
constexpr int PIPE_ST = 4;     // stages
constexpr int PIPE_MAXB = 4096;  // accepted counts cached in shared memory

struct PipeLayout {
  size_t bar, nacc, stages, stage, off_x, off_b, off_c, off_dt, rows, red, total;  // bytes
};
__host__ __device__ inline PipeLayout pipe_layout(const Dims& d, bool read) {
  PipeLayout m{};
  const int lim = d.S + 1;
  m.bar = 0;                                        // full[PIPE_ST], empty[PIPE_ST]
  m.nacc = 128;                                     // [PIPE_MAXB] counts
  m.stages = (m.nacc + (size_t)PIPE_MAXB * 4 + 127) / 128 * 128;
  m.off_x = (size_t)d.P * d.N * 4;                  // a stage: state | x rows | B rows | C rows | dt, A_log
  m.off_b = m.off_x + (size_t)lim * d.P * 4;
  m.off_c = m.off_b + (size_t)lim * d.N * 4;
  m.off_dt = m.off_c + (read ? (size_t)d.S * d.N * 4 : 0);
  m.stage = (m.off_dt + (size_t)(lim + 1) * 4 + 127) / 128 * 128;
  m.rows = m.stages + PIPE_ST * m.stage;
  m.red = m.rows + (read ? (size_t)d.P * (d.N + 8) * 4 : 0);
  m.total = m.red + (read ? (size_t)mem_ksplit(d) * d.P * 8 * 4 : 0);
  return m;
}

// A CTA's walk over items i = blockIdx.x + k * gridDim.x, kept as
// (layer, request, head) and advanced by the grid stride without divisions.
struct PipeCursor {
  int l, b, h;
  __device__ void init(int i, int Hm, int B) {
    h = i % Hm;
    b = (i / Hm) % B;
    l = i / (Hm * B);
  }
  __device__ void step(int gl, int gb, int gh, int Hm, int B) {
    h += gh;
    int cb = 0;
    if (h >= Hm) {
      h -= Hm;
      cb = 1;
    }
    b += gb + cb;
    int cl = 0;
    if (b >= B) {
      b -= B;
      cl = 1;
    }
    l += gl + cl;
  }
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// The barrier completes one of its expected arrivals once every cp.async
// this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(PIPE_THREADS)
commit_state_pipe_kernel(Dims d, int B, int early, int late, const int32_t* __restrict__ n_acc,
                         const float* __restrict__ xbd, long long xls,
                         const float* __restrict__ A_log, float* __restrict__ state,
                         int64_t* __restrict__ pos, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ tags, int32_t* __restrict__ err,
                         const float* __restrict__ memC, T* __restrict__ mix) {
  extern __shared__ __align__(128) uint8_t psm[];
  const bool rd = memC != nullptr;
  const PipeLayout L = pipe_layout(d, rd);
  uint64_t* full = reinterpret_cast<uint64_t*>(psm + L.bar);
  uint64_t* empty = full + PIPE_ST;
  int* snacc = reinterpret_cast<int*>(psm + L.nacc);
  __shared__ int s_abort;
  const int lim = d.S + 1, P = d.P, N = d.N, nq = P * N / 4;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int G = gridDim.x, gh = G % d.Hm, gb = (G / d.Hm) % B, gl = G / (d.Hm * B);
  if (!late) pdl_trigger();

  // accepted counts (the caller's input, final at launch), invalid -> 0
  for (int i = tid; i < B; i += PIPE_THREADS) {
    const int m = __ldcg(&n_acc[i]);
    snacc[i] = (m >= 0 && m <= lim) ? m : 0;
  }
  if (tid == 0) {
    for (int k = 0; k < PIPE_ST; ++k) {
      mbar_init(&full[k], 1 + 32);  // the state copy's expect_tx + the producer lanes' rows
      mbar_init(&empty[k], PIPE_CWARPS);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto next_work = [&](PipeCursor c) {  // the first item at or after c with work
    while (c.l < d.L && !(snacc[c.b] > 0 || (rd && c.l == 0))) c.step(gl, gb, gh, d.Hm, B);
    return c;
  };
  auto advance = [&](PipeCursor c) {
    c.step(gl, gb, gh, d.Hm, B);
    return next_work(c);
  };
  PipeCursor first;
  first.init(blockIdx.x, d.Hm, B);
  first = next_work(first);

  if (warp == PIPE_CWARPS) {
    // ------------------------------------------------------------ producer
    auto issue_state = [&](const PipeCursor& c, int st) {  // lane 0
      uint8_t* sg = psm + L.stages + (size_t)st * L.stage;
      const uint32_t sbytes = (uint32_t)(P * N * 4);
      mbar_expect_tx(&full[st], sbytes);
      bulk_g2s(sg, state + (((size_t)c.l * d.Bmax + c.b) * d.Hm + c.h) * (size_t)P * N, sbytes,
               &full[st]);
    };
    auto issue_rows = [&](const PipeCursor& c, int st) {  // all lanes
      const int n = snacc[c.b];
      uint8_t* sg = psm + L.stages + (size_t)st * L.stage;
      const float* xb = xbd + (size_t)c.l * xls + (size_t)c.b * lim * d.NS;
      const int px = P / 4, pb = N / 4;
      for (int e = lane; e < n * px; e += 32) {
        const int t = e / px, c4 = (e % px) * 4;
        cp_async16(sg + L.off_x + ((size_t)t * P + c4) * 4, xb + (size_t)t * d.NS + (size_t)c.h * P + c4);
      }
      for (int e = lane; e < n * pb; e += 32) {
        const int t = e / pb, c4 = (e % pb) * 4;
        cp_async16(sg + L.off_b + ((size_t)t * N + c4) * 4, xb + (size_t)t * d.NS + d.dinner + c4);
      }
      if (rd && c.l == 0)
        for (int e = lane; e < d.S * pb; e += 32) {
          const int s2 = e / pb, c4 = (e % pb) * 4;
          cp_async16(sg + L.off_c + ((size_t)s2 * N + c4) * 4, memC + ((size_t)c.b * d.S + s2) * d.Nd + c4);
        }
      if (lane < n) cp_async4(sg + L.off_dt + (size_t)lane * 4, xb + (size_t)lane * d.NS + d.dinner + N + c.h);
      if (lane == 31) cp_async4(sg + L.off_dt + (size_t)lim * 4, A_log + c.l * d.Hm + c.h);
      cp_async_arrive(&full[st]);
    };
    PipeCursor pend[PIPE_ST];
    PipeCursor cur = first;
    int npro = 0;
    for (; npro < PIPE_ST && cur.l < d.L; ++npro) {
      pend[npro] = cur;
      if (lane == 0 && early) issue_state(cur, npro);
      cur = advance(cur);
    }
    pdl_wait();
    if (late) pdl_trigger();
    for (int k = 0; k < npro; ++k) {
      if (lane == 0 && !early) issue_state(pend[k], k);
      issue_rows(pend[k], k);
    }
    // bookkeeping of the requests whose (layer 0, head 0) item this CTA owns
    for (int b = 0; b < B; ++b) {
      if ((b * d.Hm) % G != (int)blockIdx.x) continue;  // B * Hm < 2^30 (launch check)
      int part = 0;
      for (int j = lane; j < b; j += 32) part += snacc[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const int m = __ldcg(&n_acc[b]);
      const int n = snacc[b];
      const long long p0 = __ldcg(&pos[b]);
      if (lane == 0) {
        if (!(m >= 0 && m <= lim)) atomicOr(err, ERR_BAD_ACCEPTED);
        offsets[b] = part;
        if (b == B - 1) offsets[B] = part + n;
      }
      for (int t = lane; t < n; t += 32) tags[(size_t)b * d.W + (int)((p0 + t) % d.W)] = (int32_t)(p0 + t);
      __syncwarp();
      if (lane == 0) pos[b] = p0 + n;
    }
    // the rest: item j into stage j % PIPE_ST once its previous occupant
    // (item j - PIPE_ST) is released
    long long j = npro;
    long long issued = npro;
    bool ok = true;
    for (; cur.l < d.L; ++j) {
      const int st = (int)(j % PIPE_ST);
      ok = mbar_wait(&empty[st], (uint32_t)((j / PIPE_ST) & 1) ^ 1u) &&
           !*reinterpret_cast<volatile int*>(&s_abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_state(cur, st);
      }
      __syncwarp();
      issue_rows(cur, st);
      ++issued;
      cur = advance(cur);
    }
    if (!ok) {
      // a consumer gave up, or a stage was never released: report, stop
      // issuing, and let the copies of the items that may still be in
      // flight (the last PIPE_ST issued) land (bounded) before leaving
      if (lane == 0) atomicOr(err, ERR_TIMEOUT);
      for (long long q = j - PIPE_ST > 0 ? j - PIPE_ST : 0; q < issued; ++q)
        mbar_wait(&full[q % PIPE_ST], (uint32_t)(q / PIPE_ST) & 1u);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's row copies have landed
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  if (late) pdl_trigger();
  // this thread's float4 q = tid + u * PIPE_CT of a head: row pr[u], column
  // c4 (the same for every u: N / 4 divides PIPE_CT)
  const int cpr = N / 4;
  const int c4 = (tid % cpr) * 4;
  int pr[PIPE_QPT];
#pragma unroll
  for (int u = 0; u < PIPE_QPT; ++u) {
    const int q = tid + u * PIPE_CT;
    pr[u] = q < nq ? q / cpr : 0;  // elements past the head: row 0, never stored
  }
  // the fused memory read straight from the registers when every warp holds
  // whole rows (N = 128) and the head fills the threads exactly
  const bool reg_read = N == 128 && nq == PIPE_QPT * PIPE_CT && d.S <= 8 && PIPE_QPT * 8 <= 32;
  PipeCursor it = first;
  bool live = true;  // false after a wait gave up: the walk continues without work
  for (long long k = 0; it.l < d.L; ++k) {
    const int st = (int)(k % PIPE_ST);
    const int l = it.l, b = it.b, h = it.h, n = live ? snacc[b] : 0;
    if (live && (*reinterpret_cast<volatile int*>(&s_abort) ||
                 !mbar_wait(&full[st], (uint32_t)(k / PIPE_ST) & 1u))) {
      live = false;  // the producer stops issuing and drains; the named
      s_abort = 1;   // barriers below stay matched
    }
    const uint8_t* sg = psm + L.stages + (size_t)st * L.stage;
    const float4* s4 = reinterpret_cast<const float4*>(sg);
    const float* sx = reinterpret_cast<const float*>(sg + L.off_x);
    const float* sb = reinterpret_cast<const float*>(sg + L.off_b);
    const float* sdt = reinterpret_cast<const float*>(sg + L.off_dt);
    float4 hv[PIPE_QPT];
#pragma unroll
    for (int u = 0; u < PIPE_QPT; ++u) {
      const int q = tid + u * PIPE_CT;
      hv[u] = live && q < nq ? s4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // h after rows 0..n-1 of h_t = e^{dt_t A} h_{t-1} + dt_t x_t B_t^T, unrolled:
    // h_n = D h_0 + sum_t (c_t dt_t) x_t B_t^T with c_t the product of the
    // decays of the rows after t (<= 1) and D that of all n. Lane t of each
    // warp forms row t's decay; a suffix-product scan by shuffles gives c_t
    // and D, so the per-element work per row is one FMA.
    const float A = live ? -expf(sdt[lim]) : 0.f;
    float dt_l = 0.f, suf = 1.f;
    if (lane < n) {
      dt_l = sdt[lane];
      suf = expf(dt_l * A);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // suf = prod over rows >= lane
      const float v = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf *= v;
    }
    const float after = __shfl_down_sync(0xffffffffu, suf, 1);
    const float wdt = (lane < 31 ? after : 1.f) * dt_l;  // c_t dt_t at lane t
    const float D = __shfl_sync(0xffffffffu, suf, 0);
#pragma unroll
    for (int u = 0; u < PIPE_QPT; ++u) {
      hv[u].x *= D;
      hv[u].y *= D;
      hv[u].z *= D;
      hv[u].w *= D;
    }
    for (int t = 0; t < n; ++t) {
      const float w = __shfl_sync(0xffffffffu, wdt, t);
      const float4 Bv = *reinterpret_cast<const float4*>(&sb[t * N + c4]);
#pragma unroll
      for (int u = 0; u < PIPE_QPT; ++u) {
        const float xv = w * sx[t * P + pr[u]];
        hv[u].x = fmaf(xv, Bv.x, hv[u].x);
        hv[u].y = fmaf(xv, Bv.y, hv[u].y);
        hv[u].z = fmaf(xv, Bv.z, hv[u].z);
        hv[u].w = fmaf(xv, Bv.w, hv[u].w);
      }
    }
    if (live && n > 0) {
      float4* hg = reinterpret_cast<float4*>(state + (((size_t)l * d.Bmax + b) * d.Hm + h) * (size_t)P * N);
#pragma unroll
      for (int u = 0; u < PIPE_QPT; ++u) {
        const int q = tid + u * PIPE_CT;
        if (q < nq) __stcs(&hg[q], hv[u]);
      }
    }
    if (rd && l == 0 && reg_read) {
      // memory read of the new state from the registers: warp w holds rows
      // w + 16u (u < 4) whole, 4 columns per lane; per (row, slot) a partial
      // dot product over the lane's columns, then one butterfly over the
      // warp leaves lane 8u + s with y[s][row u]
      const float* sc = reinterpret_cast<const float*>(sg + L.off_c);
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2)
        if (s2 < d.S) {
          const float4 c = *reinterpret_cast<const float4*>(&sc[s2 * N + c4]);
#pragma unroll
          for (int u = 0; u < PIPE_QPT; ++u)
            v[u * 8 + s2] = hv[u].x * c.x + hv[u].y * c.y + hv[u].z * c.z + hv[u].w * c.w;
        }
      const float y = reduce_scatter32(v, lane);
      const int u = lane >> 3, sl = lane & 7;
      const int row = (tid + u * PIPE_CT) / cpr;  // pr[u], without indexing it at run time
      if (live && sl < d.S)
        mix[((size_t)b * d.S + sl) * d.Nz + d.QD + (size_t)h * P + row] = from_f<T>(y);
    } else if (rd && l == 0) {
      // memory read of the new state (tensor cores, as the per-head kernel);
      // the consumers synchronise among themselves (named barrier 1)
      const int RS = N + 8;
      float* rows = reinterpret_cast<float*>(psm + L.rows);
      float* red = reinterpret_cast<float*>(psm + L.red);
      const float* sc = reinterpret_cast<const float*>(sg + L.off_c);
#pragma unroll
      for (int u = 0; u < PIPE_QPT; ++u) {
        const int q = tid + u * PIPE_CT;
        if (live && q < nq) *reinterpret_cast<float4*>(&rows[pr[u] * RS + c4]) = hv[u];
      }
      const int g8 = lane >> 2, t4 = lane & 3;
      const int MT = P / 16, KSPL = mem_ksplit(d), G16 = N / 16 / KSPL;
      const int mt = warp % MT, kp = warp / MT;
      const bool active = live && kp < KSPL;
      const int r0 = mt * 16 + g8;
      const int col0 = kp * G16 * 16 + 4 * t4;
      asm volatile("bar.sync 1, %0;" ::"r"(PIPE_CT) : "memory");  // the new state is in rows
      if (active) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < MEM_G16; ++j)
          if (j < G16) {
            float4 cc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (g8 < d.S) cc = *reinterpret_cast<const float4*>(&sc[g8 * N + col0 + j * 16]);
            const float4 x0 = *reinterpret_cast<const float4*>(&rows[r0 * RS + col0 + j * 16]);
            const float4 x1 = *reinterpret_cast<const float4*>(&rows[(r0 + 8) * RS + col0 + j * 16]);
            mma_tf32_1688(c, to_tf32(x0.x), to_tf32(x1.x), to_tf32(x0.y), to_tf32(x1.y),
                          to_tf32(cc.x), to_tf32(cc.y));
            mma_tf32_1688(c, to_tf32(x0.z), to_tf32(x1.z), to_tf32(x0.w), to_tf32(x1.w),
                          to_tf32(cc.z), to_tf32(cc.w));
          }
        float* rp = red + ((size_t)kp * P + r0) * 8 + 2 * t4;
        *reinterpret_cast<float2*>(rp) = make_float2(c[0], c[1]);
        *reinterpret_cast<float2*>(rp + 64) = make_float2(c[2], c[3]);
      }
      asm volatile("bar.sync 1, %0;" ::"r"(PIPE_CT) : "memory");  // partial sums in red
      for (int e = live ? tid : d.S * P; e < d.S * P; e += PIPE_CT) {
        const int sl = e / P, p = e % P;
        float y = 0.f;
        for (int q = 0; q < KSPL; ++q) y += red[((size_t)q * P + p) * 8 + sl];
        mix[((size_t)b * d.S + sl) * d.Nz + d.QD + (size_t)h * P + p] = from_f<T>(y);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with stage st
    it = advance(it);
  }
}

}  // namespace

size_t commit_state_smem(const Dims& d, bool read) { return cs_layout(d, read).total * sizeof(float); }

namespace {
template <typename K>
cudaError_t set_smem(K kernel, int smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int R>
cudaError_t configure_variant(int smem) {
  cudaError_t e = set_smem(commit_state_kernel<float, 2, R>, smem);
  if (e == cudaSuccess) e = set_smem(commit_state_kernel<float, QPT_HEAD, R>, smem);
  if (e == cudaSuccess) e = set_smem(commit_state_kernel<__nv_bfloat16, 2, R>, smem);
  if (e == cudaSuccess) e = set_smem(commit_state_kernel<__nv_bfloat16, QPT_HEAD, R>, smem);
  return e;
}

template <int R>
cudaError_t launch_variant(int dtype, const Dims& d, int B, bool whole, int qsplit, size_t smem,
                           int early, int late, const int32_t* n_acc, const float* xbd,
                           long long xls, const float* A_log, float* state, int64_t* pos,
                           int32_t* offsets, int32_t* tags, int32_t* err, const float* memC,
                           void* mix, const MemRing& mr, cudaStream_t st) {
  const dim3 grid(d.Hm * qsplit, B, d.L);
  const dim3 blk(THREADS_CS);
  if (dtype == HF_F32) {
    auto k = whole ? commit_state_kernel<float, QPT_HEAD, R> : commit_state_kernel<float, 2, R>;
    return launch_pdl(k, grid, blk, smem, st, d, B, qsplit, early, late, n_acc, xbd, xls, A_log,
                      state, pos, offsets, tags, err, memC, (float*)mix, mr);
  }
  auto k = whole ? commit_state_kernel<__nv_bfloat16, QPT_HEAD, R>
                 : commit_state_kernel<__nv_bfloat16, 2, R>;
  return launch_pdl(k, grid, blk, smem, st, d, B, qsplit, early, late, n_acc, xbd, xls, A_log,
                    state, pos, offsets, tags, err, memC, (__nv_bfloat16*)mix, mr);
}
}  // namespace

// The kernels' shared-memory attribute is a per-device setting: keep, per
// device, the largest need configured so far.
constexpr int kMaxDevices = 64;
std::mutex g_cs_mu;
int g_cs_configured[kMaxDevices] = {}, g_cs_configured_pipe[kMaxDevices] = {};

cudaError_t configure_commit_state(const Dims& d) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_cs_mu);
  const int smem = (int)commit_state_smem(d, mem_tc_ok(d));
  if (smem > g_cs_configured[dev]) {
    e = configure_variant<0>(smem);
    if (e == cudaSuccess) e = configure_variant<1>(smem);
    if (e == cudaSuccess) e = configure_variant<2>(smem);
    if (e == cudaSuccess) g_cs_configured[dev] = smem;
  }
  const int psmem = (int)pipe_layout(d, mem_tc_ok(d)).total;
  if (e == cudaSuccess && psmem > g_cs_configured_pipe[dev] && psmem <= 232448) {
    e = set_smem(commit_state_pipe_kernel<float>, psmem);
    if (e == cudaSuccess) e = set_smem(commit_state_pipe_kernel<__nv_bfloat16>, psmem);
    if (e == cudaSuccess) g_cs_configured_pipe[dev] = psmem;
  }
  return e;
}

cudaError_t launch_commit_state(int dtype, const Dims& d, int B, const int32_t* n_acc,
                                const float* xbd, long long xls, const float* A_log, float* state,
                                int64_t* pos, int32_t* offsets, int32_t* tags, int32_t* err,
                                const float* memC, void* mix, int early, int late,
                                int num_sms, const MemRing& mr, cudaStream_t st) {
  if (memC && (dtype != HF_BF16 || !mem_tc_ok(d))) return cudaErrorInvalidValue;
  if (d.Mr > 0 && (!mr.x || !mr.b || !mr.dt || !mr.pos_snap)) return cudaErrorInvalidValue;
  const int nq = d.P * d.N / 4;
  if (nq > QPT_HEAD * THREADS_CS) return cudaErrorInvalidValue;
  // whole heads per CTA when fused or when they alone give ~4 CTAs per SM
  const bool whole = memC != nullptr || (long long)B * d.Hm * d.L >= 4LL * num_sms;
  const int qpt = whole ? QPT_HEAD : 2;
  const int qsplit = (nq + qpt * THREADS_CS - 1) / (qpt * THREADS_CS);
  const size_t smem = commit_state_smem(d, memC != nullptr);
  // large batches of the plain Mamba-2 memory: the pipelined persistent walk
  const PipeLayout pl = pipe_layout(d, memC != nullptr);
  if (!d.gdn && d.Mr == 0 && d.Mh == 0 && whole && pl.total <= 232448 && d.S + 1 <= 32 &&
      nq <= PIPE_QPT * PIPE_THREADS && B <= PIPE_MAXB &&
      (long long)B * d.Hm * d.L >= 8LL * num_sms && (long long)B * d.Hm * d.L < (1LL << 30)) {
    const long long items = (long long)B * d.Hm * d.L;
    const dim3 grid((unsigned)std::min<long long>(num_sms, items));
    if (dtype == HF_F32)
      return launch_pdl(commit_state_pipe_kernel<float>, grid, dim3(PIPE_THREADS), pl.total, st, d,
                        B, early, late, n_acc, xbd, xls, A_log, state, pos, offsets, tags, err,
                        memC, (float*)mix);
    return launch_pdl(commit_state_pipe_kernel<__nv_bfloat16>, grid, dim3(PIPE_THREADS), pl.total,
                      st, d, B, early, late, n_acc, xbd, xls, A_log, state, pos, offsets, tags,
                      err, memC, (__nv_bfloat16*)mix);
  }
  if (d.gdn)
    return launch_variant<2>(dtype, d, B, whole, qsplit, smem, early, late, n_acc, xbd, xls, A_log,
                             state, pos, offsets, tags, err, memC, mix, mr, st);
  if (d.Mr > 0)
    return launch_variant<1>(dtype, d, B, whole, qsplit, smem, early, late, n_acc, xbd, xls, A_log,
                             state, pos, offsets, tags, err, memC, mix, mr, st);
  return launch_variant<0>(dtype, d, B, whole, qsplit, smem, early, late, n_acc, xbd, xls, A_log,
                           state, pos, offsets, tags, err, memC, mix, mr, st);
}

cudaError_t launch_gdn_prefill(const Dims& d, int layer, int b, int T, const float* xs,
                               const float* A_log, float* state, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int nq = d.P * d.N / 4;
  const int qsplit = (nq + QPT_SCAN * THREADS_CS - 1) / (QPT_SCAN * THREADS_CS);
  gdn_prefill_kernel<<<d.Hm * qsplit, THREADS_CS, 0, st>>>(d, layer, b, T, qsplit, xs, A_log,
                                                            state);
  return cudaGetLastError();
}

}  // namespace hf
