// Host runtime and C ABI of the HyFlash drafter-layer library.
//
// The handle owns, per layer, the window rings and recurrent states of all
// requests, the re-laid-out weights, and the scratch the kernels need. Every
// call enqueues kernels on the caller's stream; host work is argument
// checking, pointer arithmetic and grid sizing only.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

using hf::Dims;
using hf::Epi;

struct ProfRec {
  cudaEvent_t a, b;
  int fam;
  int count;
};

struct hf_handle {
  hf_config cfg{};
  int device = 0;
  Dims d{};
  size_t esz = 4;
  std::vector<void*> allocs;   // what cudaMalloc returned (guard region first)
  std::vector<size_t> alloc_bytes;  // usable bytes of each, between its guards

  void* w_draft = nullptr;   // [L][Nd][D]
  void* w_commit = nullptr;  // [L][Nc][D]
  void* w_out = nullptr;     // [L][D][Nz]
  // bf16: the same three weights pre-tiled for the tensor-core GEMM
  // (tile_weights; commit weights padded per layer to a multiple of 128 rows)
  void* wt_draft = nullptr;
  void* wt_commit = nullptr;
  void* wt_out = nullptr;
  int q4 = 0;  // weight_bits = 4: the wt_* tiles hold 4-bit tiles (tile_weights_q4)
  size_t wt_draft_l = 0, wt_commit_l = 0, wt_out_l = 0;  // bytes per layer
  int nc_pad = 0;                                         // padded commit rows per layer
  float* dt_bias = nullptr;  // [L][Hm]
  float* A_log = nullptr;    // [L][Hm]

  void* ring_k = nullptr;    // [L][Bmax][Hkv][W][dh]
  void* ring_v = nullptr;
  int32_t* tags = nullptr;   // [Bmax][W]
  int64_t* pos = nullptr;    // [Bmax]
  float* state = nullptr;    // [L][Bmax][Hm][P][N]
  // memory horizon M > 1: x / B / dt of the last M + S + 1 committed features
  float* mem_x = nullptr;    // [L][Bmax][Mr][dinner]
  float* mem_b = nullptr;    // [L][Bmax][Mr][N]
  float* mem_dt = nullptr;   // [L][Bmax][Hm][Mr]
  int64_t* pos_snap = nullptr;  // [Bmax]: positions before the running commit
  int64_t* req_len = nullptr;   // [Bmax]: prefix lengths of the running prefill
  float* gdn_xs = nullptr;      // gated delta: x | B | dt | beta of a prefill pass [Tseg][NS]

  int32_t* offsets = nullptr;  // [Bmax+1]
  int32_t* row_req = nullptr;  // [Rmax]
  int64_t* row_pos = nullptr;  // [Rmax]
  void* packed = nullptr;      // [Rmax][D]
  long long rmax = 0;
  float* xbd = nullptr;        // [L][(S+1)*Bmax][NS]
  long long xbd_ls = 0;

  float* proj = nullptr;       // [Bmax*S][Nd]
  void* mix = nullptr;         // [Bmax*S][Nz]
  void* xbuf[2] = {nullptr, nullptr};
  float* part = nullptr;
  size_t part_elems = 0;
  std::vector<CUtensorMap> ring_maps;  // per layer: K, V tile maps (tensor-core attention)
  std::vector<CUtensorMap> state_maps; // per layer: the memory states (its memory-read CTAs)
  int* counters = nullptr;     // tile tickets of the stream-K GEMM (zero between launches)
  int n_counters = 0;
  float* skws = nullptr;       // stream-K partial tiles
  size_t skws_floats = 0;
  int num_sms = 152;

  // prefill segment scratch (Tseg = pf_tokens tokens, transposed layouts)
  float* pf_dtw = nullptr;     // [Hm][Tseg] fp32: dt, then decay weights w
  float* pf_decay = nullptr;   // [Hm] fp32: decay of the whole segment
  void* pf_xsT = nullptr;      // [Hm*P][Tseg] model dtype: w * x
  void* pf_bT = nullptr;       // [N][Tseg] model dtype: B
  long long pf_tokens = 0;
  int32_t* pf_lens = nullptr;  // [Bmax]
  int32_t* pf_reqs = nullptr;  // [Bmax]

  int32_t* err = nullptr;

  // full drafter block (block_kind = 1)
  float* g_mix = nullptr;      // [L][D]
  float* g_mlp = nullptr;      // [L][D]
  float* d_skip = nullptr;     // [L][Hm]
  float* conv_w = nullptr;     // [L][C][4], C = dinner + N
  float* conv_b = nullptr;     // [L][C]
  float* conv_state = nullptr; // [L][Bmax][3][C]: last 3 pre-conv committed rows
  void* w_up = nullptr;        // [L][2F][D]: W_gate^T rows, then W_up^T rows
  void* w_down = nullptr;      // [L][D][F]
  void* wt_up = nullptr;       // bf16 tiles of the same
  void* wt_down = nullptr;
  size_t wt_up_l = 0, wt_down_l = 0;
  float* g_final = nullptr;    // [D]
  void* w_lm = nullptr;        // [V][D]
  void* wt_lm = nullptr;
  int head_set = 0;
  void* anorm = nullptr;       // [Bmax*S][D]: normed rows (model dtype)
  void* x1 = nullptr;          // [Bmax*S][D]: X + mixer branches
  float* mlp_h = nullptr;      // [Bmax*S][2F]: gate | up
  void* act = nullptr;         // [Bmax*S][F]
  float* logits = nullptr;     // [Bmax*S][V]
  float* pf_u = nullptr;       // [Tseg][C]: pre-conv x | B rows of a prefill pass
  double* rope_inv = nullptr;  // [dh/2]: theta^(-2i/dh)

  int prof = 0;                 // 0 off, 1 records read once, 2 records kept (graphs)
  std::vector<ProfRec> pending;  // mode 1
  std::vector<ProfRec> kept;     // mode 2
  std::vector<cudaEvent_t> pool;
  double tot_ms[HF_K_COUNT] = {};
  int64_t nl[HF_K_COUNT] = {};
  int64_t launches = 0;
  std::string msg;
};

namespace {

thread_local std::string g_create_error;

hf_status fail(hf_handle* h, hf_status s, const std::string& m) {
  if (h) h->msg = m;
  else g_create_error = m;
  return s;
}

hf_status cuda_fail(hf_handle* h, cudaError_t e, const char* where) {
  return fail(h, HF_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define HF_CUDA(h, call)                                  \
  do {                                                    \
    cudaError_t _e = (call);                              \
    if (_e != cudaSuccess) return cuda_fail(h, _e, #call); \
  } while (0)

long long round_up(long long a, long long b) { return (a + b - 1) / b * b; }

Dims make_dims(const hf_config& c) {
  Dims d{};
  d.D = c.d_model; d.Hq = c.n_q_heads; d.Hkv = c.n_kv_heads; d.dh = c.head_dim;
  d.W = c.window; d.S = c.block; d.Hm = c.ssm_heads; d.P = c.ssm_headdim; d.N = c.d_state;
  d.L = c.n_layers; d.Bmax = c.max_batch;
  d.G = d.Hq / d.Hkv;
  d.QD = d.Hq * d.dh;
  d.KVD = d.Hkv * d.dh;
  d.dinner = d.Hm * d.P;
  d.Nd = d.QD + 2 * d.KVD + d.N;
  d.gdn = c.memory_kind == HF_MEM_GATED_DELTA ? 1 : 0;
  d.Nc = 2 * d.KVD + d.dinner + d.N + d.Hm * (1 + d.gdn);  // [K | V | x | B | dt (| beta)]
  d.NS = (int)round_up(d.dinner + d.N + d.Hm * (1 + d.gdn), 4);
  d.Nz = d.QD + d.dinner;
  d.esize = c.dtype == HF_F32 ? 4 : 2;
  d.xoff = c.cross_slot_off ? 1 : 0;
  d.Mh = c.mem_horizon;
  d.Mr = c.mem_horizon > 1 ? c.mem_horizon + c.block + 1 : 0;
  d.wait = hf::kWaitCycles;
  d.blk = c.block_kind == HF_FULL_BLOCK ? 1 : 0;
  d.F = d.blk ? c.mlp_dim : 0;
  d.V = d.blk ? c.vocab : 0;
  if (d.blk) d.Nd += 2 * d.dinner;  // + x_s | z_s (skip and gate of the memory read)
  return d;
}

hf_status validate(const hf_config* c, std::string* why) {
  auto bad = [&](const char* m) { *why = m; return HF_EINVAL; };
  if (!c) return bad("config is NULL");
  if (c->d_model <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->window <= 0 || c->block <= 0 || c->ssm_heads <= 0 || c->ssm_headdim <= 0 ||
      c->d_state <= 0 || c->n_layers <= 0 || c->max_batch <= 0)
    return bad("every dimension must be positive");
  if (c->n_groups != 1) return bad("n_groups must be 1");
  if (c->n_q_heads % c->n_kv_heads) return bad("n_kv_heads must divide n_q_heads");
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
    return bad("head_dim must be 32, 64, 128 or 256");
  if (c->d_state < 4 || c->d_state > 128 || (c->d_state & (c->d_state - 1)))
    return bad("d_state must be a power of two in 4..128");
  if (c->ssm_headdim % 4) return bad("ssm_headdim must be a multiple of 4");
  if ((long long)c->ssm_headdim * c->d_state > 8192 || ((long long)c->ssm_headdim * c->d_state) % 128)
    return bad("ssm_headdim * d_state must be a multiple of 128, <= 8192");
  if (c->block > 16) return bad("block must be <= 16");
  if (c->window < c->block + 1) return bad("window must be >= block + 1");
  if ((c->n_q_heads / c->n_kv_heads) * c->block > 64) return bad("(n_q_heads/n_kv_heads)*block must be <= 64");
  if (c->chunk != 64 && c->chunk != 128 && c->chunk != 256) return bad("chunk must be 64, 128 or 256");
  if (c->dtype != HF_F32 && c->dtype != HF_BF16) return bad("dtype must be HF_F32 or HF_BF16");
  if (c->d_model % 8) return bad("d_model must be a multiple of 8");
  if (c->prefill_tokens_max < 0) return bad("prefill_tokens_max must be >= 0");
  if (c->max_batch > 65535) return bad("max_batch must be <= 65535");
  if (c->dtype == HF_BF16 && c->ssm_headdim % 16)
    return bad("bf16 needs ssm_headdim a multiple of 16");
  if (c->cross_slot_off != 0 && c->cross_slot_off != 1) return bad("cross_slot_off must be 0 or 1");
  if (c->mem_horizon < 0 || c->mem_horizon > c->window)
    return bad("mem_horizon must be in 0..window");
  if (c->memory_kind != HF_MEM_MAMBA2 && c->memory_kind != HF_MEM_GATED_DELTA)
    return bad("memory_kind must be HF_MEM_MAMBA2 or HF_MEM_GATED_DELTA");
  if (c->memory_kind == HF_MEM_GATED_DELTA && c->mem_horizon != 0)
    return bad("the gated-delta memory takes no memory horizon");
  if (c->weight_bits != 0 && c->weight_bits != 16 && c->weight_bits != 4)
    return bad("weight_bits must be 16 or 4");
  if (c->weight_bits == 4) {
    if (c->dtype != HF_BF16) return bad("4-bit weights need a bf16 handle");
    if (c->d_model % 128 || ((long long)c->n_q_heads * c->head_dim) % 128 ||
        ((long long)c->ssm_heads * c->ssm_headdim) % 128)
      return bad("4-bit weights need d_model, n_q_heads*head_dim, ssm_heads*ssm_headdim multiples of 128");
  }
  if (c->block_kind != HF_LAYER && c->block_kind != HF_FULL_BLOCK)
    return bad("block_kind must be HF_LAYER or HF_FULL_BLOCK");
  if (c->block_kind == HF_FULL_BLOCK) {
    if (c->memory_kind != HF_MEM_MAMBA2 || c->mem_horizon != 0)
      return bad("the full block takes the Mamba-2 memory without a horizon");
    if (c->weight_bits == 4) return bad("the full block takes weight_bits 16");
    if (c->mlp_dim < 8 || c->mlp_dim % 8) return bad("mlp_dim must be a positive multiple of 8");
    if (c->vocab < 2) return bad("vocab must be >= 2");
    if (c->head_dim % 2) return bad("head_dim must be even (RoPE pairs)");
  }
  {
    const Dims d = make_dims(*c);
    if (hf::attn_cluster_smem(d, d.esize) > 232448)
      return bad("window too long for the attention tile (shared memory per CTA > 227 KB)");
  }
  return HF_OK;
}

// Test hook: the k-th device allocation from now on fails as if the device
// were out of memory (0: off).
std::atomic<long long> g_fail_alloc_in{0};

// Every buffer sits between two guard regions of kGuardBytes filled with
// kGuardByte; hf_debug_check_guards reads them back. The usable part starts
// kGuardBytes after cudaMalloc's (256-byte aligned) address.
constexpr size_t kGuardBytes = 256;
constexpr int kGuardByte = 0xA5;

hf_status dev_alloc(hf_handle* h, void** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  bytes = (bytes + 255) / 256 * 256;
  long long k = g_fail_alloc_in.load();
  while (k > 0 && !g_fail_alloc_in.compare_exchange_weak(k, k - 1)) {
  }
  void* base = nullptr;
  cudaError_t e = k == 1 ? cudaErrorMemoryAllocation : cudaMalloc(&base, bytes + 2 * kGuardBytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(h, HF_ENOMEM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed: " +
                                  cudaGetErrorString(e));
  }
  h->allocs.push_back(base);
  h->alloc_bytes.push_back(bytes);
  *p = static_cast<char*>(base) + kGuardBytes;
  e = cudaMemset(base, kGuardByte, kGuardBytes);
  if (e == cudaSuccess) e = cudaMemset(*p, 0, bytes);
  if (e == cudaSuccess) e = cudaMemset(static_cast<char*>(*p) + bytes, kGuardByte, kGuardBytes);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemset");
  return HF_OK;
}

void free_all(hf_handle* h) {
  for (auto* v : {&h->pending, &h->kept})
    for (auto& r : *v) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
  h->kept.clear();
  for (auto e : h->pool) cudaEventDestroy(e);
  h->pending.clear();
  h->pool.clear();
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
  h->alloc_bytes.clear();
}

// ---- profiling: events around launches of one family
cudaEvent_t get_event(hf_handle* h) {
  if (!h->pool.empty()) {
    cudaEvent_t e = h->pool.back();
    h->pool.pop_back();
    return e;
  }
  cudaEvent_t e;
  cudaEventCreate(&e);
  return e;
}

struct Scope {
  hf_handle* h;
  int fam;
  cudaStream_t st;
  ProfRec rec{};
  int before;
  int count = 0;  // launches made inside the scope
  // Mode 2 records with cudaEventRecordExternal so that, inside stream
  // capture, the records become graph nodes that re-record on every replay.
  unsigned flags() const { return h->prof == 2 ? cudaEventRecordExternal : cudaEventRecordDefault; }
  Scope(hf_handle* h_, int fam_, cudaStream_t st_) : h(h_), fam(fam_), st(st_) {
    if (h->prof) {
      rec.a = get_event(h);
      rec.b = get_event(h);
      rec.fam = fam;
      cudaEventRecordWithFlags(rec.a, st, flags());
    }
  }
  ~Scope() {
    h->launches += count;
    if (h->prof) {
      cudaEventRecordWithFlags(rec.b, st, flags());
      rec.count = count;
      (h->prof == 2 ? h->kept : h->pending).push_back(rec);
    }
  }
};

// Add the elapsed time of every finished record to the family totals. Mode-1
// records are released; mode-2 records stay (their events are re-recorded by
// each replay of the graph they were captured into).
hf_status collect_profile(hf_handle* h) {
  for (auto* v : {&h->pending, &h->kept}) {
    if (v->empty()) continue;
    cudaError_t e = cudaEventSynchronize(v->back().b);
    if (e != cudaSuccess) {
      cudaGetLastError();
      continue;  // never recorded yet (a captured graph not replayed)
    }
    for (auto& r : *v) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
        h->tot_ms[r.fam] += ms;
        h->nl[r.fam] += r.count;
      } else {
        cudaGetLastError();
      }
    }
  }
  for (auto& r : h->pending) {
    h->pool.push_back(r.a);
    h->pool.push_back(r.b);
  }
  h->pending.clear();
  return HF_OK;
}

// Current device switch only when needed (cheap, and legal during capture).
cudaError_t ensure_device(const hf_handle* h) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return e;
  return cur == h->device ? cudaSuccess : cudaSetDevice(h->device);
}

int pick_splits(const hf_handle* h, long long R, long long C, long long K, int tile_r, int tile_c) {
  long long tiles = ((R + tile_r - 1) / tile_r) * ((C + tile_c - 1) / tile_c);
  int s = (int)std::max<long long>(1, (2 * 152 + tiles - 1) / tiles);
  s = (int)std::min<long long>(s, std::max<long long>(1, K / 256));
  s = std::min(s, 16);
  while (s > 1 && (size_t)s * R * C > h->part_elems) --s;
  return s;
}

// Y[r, c] = sum_k X[r, k] Wt[c, k] with epilogue. fp32 handles use the
// CUDA-core kernel; bf16 handles use the tensor-core kernel with the weights
// as the 128-row operand (they stream once) and the activation rows as N.
cudaError_t gemm_launch(hf_handle* h, const void* X, int ldx, const void* Wt, int ldw, int R,
                        int C, int K, const Epi& epi, cudaStream_t st, int* count,
                        const void* tiles = nullptr, int late_trigger = 0, int tile_group = 0) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (h->cfg.dtype == HF_F32) {
    int splits = pick_splits(h, R, C, K, 64, 64);
    return hf::launch_gemm_fma(h->cfg.dtype, X, ldx, Wt, ldw, R, C, K, splits, h->part, epi, st,
                               count);
  }
  // more than 32 rows: token-major (contiguous epilogue runs); products with
  // at least a tile per SM run on the persistent kernel (two accumulators,
  // epilogue overlapped, grouped tile order), smaller ones as split-K
  // partners in a cluster summing through distributed shared memory
  if (R > 32 && C >= 256 && (long long)((R + 127) / 128) * ((C + 255) / 256) >= h->num_sms &&
      !late_trigger)
    return hf::launch_gemm_persistent(X, ldx, R, Wt, ldw, C, K, h->err, epi, h->num_sms, st, count);
  if (R > 32)
    return hf::launch_gemm_tc(X, ldx, R, Wt, ldw, C, K, 0, hf::tc_pick_splits(R, C, K), h->err,
                              epi, st, count, nullptr, late_trigger);
  // skinny and more weight tiles than SMs: stream-K (no partial last wave);
  // otherwise one CTA or split-K cluster per tile (measured faster there)
  if (tiles && R <= 32 && (C + 127) / 128 > h->num_sms && !h->q4)
    return hf::launch_gemm_sk(tiles, C, tile_group, X, ldx, R, epi, nullptr, 0, nullptr, 0, 0, epi,
                              K, h->num_sms, h->skws, h->skws_floats, h->counters, h->n_counters,
                              h->err, late_trigger, st, count);
  const int splits = hf::tc_pick_splits(C, R, K, tiles && h->q4 ? 1 : 0);
  return hf::launch_gemm_tc(Wt, ldw, C, X, ldx, R, K, 1, splits, h->err, epi, st, count, tiles,
                            late_trigger, tile_group, tiles && h->q4 ? 1 : 0);
}

hf_status gemm(hf_handle* h, int fam, const void* X, int ldx, const void* Wt, int ldw, int R,
               int C, int K, const Epi& epi, cudaStream_t st, const void* tiles = nullptr,
               int late_trigger = 0, int tile_group = 0) {
  if (R <= 0 || C <= 0) return HF_OK;
  Scope sc(h, fam, st);
  cudaError_t e =
      gemm_launch(h, X, ldx, Wt, ldw, R, C, K, epi, st, &sc.count, tiles, late_trigger, tile_group);
  if (e != cudaSuccess) return cuda_fail(h, e, "gemm launch");
  return HF_OK;
}

// Y[t, c] = sum_k F[t, k] W[c, k] over the T tokens of a prefill segment,
// tokens as the 128-row operand (no split: T is large), epilogue per element.
cudaError_t tokens_gemm(hf_handle* h, const void* F, int T, const void* W, int C, const Epi& epi,
                        cudaStream_t st, int* count) {
  const Dims& d = h->d;
  if (h->cfg.dtype == HF_F32)
    return hf::launch_gemm_fma(h->cfg.dtype, F, d.D, W, d.D, T, C, d.D, 1, h->part, epi, st, count);
  if (C >= 256 && (long long)((T + 127) / 128) * ((C + 255) / 256) >= h->num_sms)
    return hf::launch_gemm_persistent(F, d.D, T, W, d.D, C, d.D, h->err, epi, h->num_sms, st, count);
  return hf::launch_gemm_tc(F, d.D, T, W, d.D, C, d.D, 0, 1, h->err, epi, st, count);
}

Epi epi_base(const hf_handle* h) {
  Epi e{};
  e.d = h->d;
  e.dt_bias = h->dt_bias;
  e.ring_k = h->ring_k;
  e.ring_v = h->ring_v;
  return e;
}

char* bptr(void* p, size_t off) { return static_cast<char*>(p) + off; }
const char* bptr(const void* p, size_t off) { return static_cast<const char*>(p) + off; }

}  // namespace

namespace hf {
void set_thread_error(const char* msg) { g_create_error = msg ? msg : ""; }
}  // namespace hf

extern "C" {

const char* hf_status_string(hf_status s) {
  switch (s) {
    case HF_OK: return "HF_OK";
    case HF_EINVAL: return "HF_EINVAL";
    case HF_ENOMEM: return "HF_ENOMEM";
    case HF_ECUDA: return "HF_ECUDA";
    case HF_ETIMEOUT: return "HF_ETIMEOUT";
    case HF_EDEVICE: return "HF_EDEVICE";
  }
  return "HF_UNKNOWN";
}

const char* hf_last_error(const hf_handle* h) {
  return h ? h->msg.c_str() : g_create_error.c_str();
}

hf_status hf_create(const hf_config* cfg, int32_t device, hf_handle** out) {
  if (!out) return fail(nullptr, HF_EINVAL, "out is NULL");
  *out = nullptr;
  std::string why;
  if (validate(cfg, &why) != HF_OK) return fail(nullptr, HF_EINVAL, why);
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return fail(nullptr, HF_ECUDA, std::string("no CUDA device: ") + cudaGetErrorString(e));
  }
  if (device < 0 || device >= ndev) return fail(nullptr, HF_EINVAL, "device index out of range");
  e = cudaSetDevice(device);
  if (e != cudaSuccess) return fail(nullptr, HF_ECUDA, cudaGetErrorString(e));

  hf_handle* h = new hf_handle();
  h->cfg = *cfg;
  if (h->cfg.prefill_tokens_max == 0) h->cfg.prefill_tokens_max = 16384;
  h->device = device;
  h->d = make_dims(h->cfg);
  const Dims& d = h->d;
  h->esz = d.esize;
  const size_t es = h->esz;
  const size_t L = d.L, Bm = d.Bmax;
  h->rmax = std::max<long long>((long long)(d.S + 1) * Bm, (long long)Bm * d.W);
  h->xbd_ls = (long long)(d.S + 1) * Bm * d.NS;
  h->pf_tokens = round_up(h->cfg.prefill_tokens_max, 64);
  h->part_elems = (size_t)16 << 20;

  hf_status s = HF_OK;
  auto A = [&](void** p, size_t bytes) {
    if (s == HF_OK) s = dev_alloc(h, p, bytes);
  };
  A(&h->w_draft, L * d.Nd * d.D * es);
  A(&h->w_commit, L * d.Nc * d.D * es);
  A(&h->w_out, L * d.D * d.Nz * es);
  if (h->cfg.dtype == HF_BF16) {
    h->nc_pad = (d.Nc + 127) / 128 * 128;
    h->q4 = h->cfg.weight_bits == 4 ? 1 : 0;
    h->wt_draft_l = h->q4 ? hf::q4_tiled_bytes(d.Nd, d.D) : hf::tiled_bytes(d.Nd, d.D);
    h->wt_commit_l = h->q4 ? hf::q4_tiled_bytes(h->nc_pad, d.D) : hf::tiled_bytes(h->nc_pad, d.D);
    h->wt_out_l = h->q4 ? hf::q4_tiled_bytes(d.D, d.Nz) : hf::tiled_bytes(d.D, d.Nz);
    A(&h->wt_draft, L * h->wt_draft_l);
    A(&h->wt_commit, L * h->wt_commit_l);
    A(&h->wt_out, L * h->wt_out_l);
  }
  A((void**)&h->dt_bias, L * d.Hm * 4);
  A((void**)&h->A_log, L * d.Hm * 4);
  A(&h->ring_k, L * Bm * d.Hkv * d.W * d.dh * es);
  A(&h->ring_v, L * Bm * d.Hkv * d.W * d.dh * es);
  A((void**)&h->tags, Bm * d.W * 4);
  A((void**)&h->pos, Bm * 8);
  A((void**)&h->state, L * Bm * d.Hm * d.P * d.N * 4);
  if (d.Mr > 0) {
    A((void**)&h->mem_x, L * Bm * d.Mr * d.dinner * 4);
    A((void**)&h->mem_b, L * Bm * d.Mr * d.N * 4);
    A((void**)&h->mem_dt, L * Bm * d.Hm * d.Mr * 4);
    A((void**)&h->pos_snap, Bm * 8);
    A((void**)&h->req_len, Bm * 8);
  }
  A((void**)&h->offsets, (Bm + 1) * 4);
  A((void**)&h->row_req, h->rmax * 4);
  A((void**)&h->row_pos, h->rmax * 8);
  A(&h->packed, h->rmax * d.D * es);
  A((void**)&h->xbd, L * h->xbd_ls * 4);
  A((void**)&h->proj, Bm * d.S * d.Nd * 4);
  A(&h->mix, Bm * d.S * d.Nz * es);
  A(&h->xbuf[0], Bm * d.S * d.D * es);
  A(&h->xbuf[1], Bm * d.S * d.D * es);
  A((void**)&h->part, h->part_elems * 4);
  h->n_counters = 1 << 16;
  A((void**)&h->counters, (size_t)h->n_counters * 4);
  if (s == HF_OK) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess && sms > 0)
      h->num_sms = sms;
  }
  if (h->cfg.dtype == HF_BF16) {
    // stream-K workspace for the largest skinny product: slot projections,
    // output projections, commit projections (alone or grouped with the
    // first slot projection)
    int tiles = 0, nslot = 0;
    size_t need = hf::gemm_sk_workspace(d.Nd, 0, d.D, h->num_sms, &tiles, &nslot);
    need = std::max(need, hf::gemm_sk_workspace(d.D, 0, d.Nz, h->num_sms, &tiles, &nslot));
    need = std::max(need, hf::gemm_sk_workspace(d.L * h->nc_pad, d.Nd, d.D, h->num_sms, &tiles, &nslot));
    need = std::max(need, hf::gemm_tm_workspace(h->num_sms));
    if (d.blk) {
      need = std::max(need, hf::gemm_sk_workspace(2 * d.F, 0, d.D, h->num_sms, &tiles, &nslot));
      need = std::max(need, hf::gemm_sk_workspace(d.D, 0, d.F, h->num_sms, &tiles, &nslot));
      need = std::max(need, hf::gemm_sk_workspace(d.V, 0, d.D, h->num_sms, &tiles, &nslot));
    }
    h->skws_floats = need;
    A((void**)&h->skws, need * 4);
  }
  if (d.gdn) A((void**)&h->gdn_xs, (size_t)h->pf_tokens * d.NS * 4);
  if (d.blk) {
    const size_t C = d.dinner + d.N, rows = Bm * d.S;
    A((void**)&h->g_mix, L * d.D * 4);
    A((void**)&h->g_mlp, L * d.D * 4);
    A((void**)&h->d_skip, L * d.Hm * 4);
    A((void**)&h->conv_w, L * C * 4 * 4);
    A((void**)&h->conv_b, L * C * 4);
    A((void**)&h->conv_state, L * Bm * 3 * C * 4);
    A(&h->w_up, L * 2 * d.F * d.D * es);
    A(&h->w_down, L * d.D * d.F * es);
    A((void**)&h->g_final, d.D * 4);
    A(&h->w_lm, (size_t)d.V * d.D * es);
    if (h->cfg.dtype == HF_BF16) {
      h->wt_up_l = hf::tiled_bytes(2LL * d.F, d.D);
      h->wt_down_l = hf::tiled_bytes(d.D, d.F);
      A(&h->wt_up, L * h->wt_up_l);
      A(&h->wt_down, L * h->wt_down_l);
      A(&h->wt_lm, hf::tiled_bytes(d.V, d.D));
    }
    A(&h->anorm, rows * d.D * es);
    A(&h->x1, rows * d.D * es);
    A((void**)&h->mlp_h, rows * 2 * d.F * 4);
    A(&h->act, rows * d.F * es);
    A((void**)&h->logits, rows * d.V * 4);
    A((void**)&h->pf_u, (size_t)h->pf_tokens * C * 4);
    A((void**)&h->rope_inv, (size_t)(d.dh / 2) * 8);
    if (s == HF_OK) {
      std::vector<double> inv(d.dh / 2);
      for (int i = 0; i < d.dh / 2; ++i) inv[i] = std::pow(1e6, -2.0 * i / d.dh);
      e = cudaMemcpy(h->rope_inv, inv.data(), inv.size() * 8, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) s = cuda_fail(h, e, "cudaMemcpy(rope table)");
    }
  }
  A((void**)&h->pf_dtw, (size_t)d.Hm * h->pf_tokens * 4);
  A((void**)&h->pf_decay, (size_t)d.Hm * 4);
  A(&h->pf_xsT, (size_t)d.dinner * h->pf_tokens * es);
  A(&h->pf_bT, (size_t)d.N * h->pf_tokens * es);
  A((void**)&h->pf_lens, Bm * 4);
  A((void**)&h->pf_reqs, Bm * 4);
  A((void**)&h->err, 16);
  if (s == HF_OK) {
    // Empty ring slots carry tag -1.
    e = cudaMemset(h->tags, 0xff, Bm * d.W * 4);
    if (e != cudaSuccess) s = cuda_fail(h, e, "cudaMemset(tags)");
  }
  if (s == HF_OK && hf::attn_uses_tc(d, h->cfg.dtype)) {
    // 2-D maps over each layer's rings: rows = Bmax*Hkv*W, box = one attention tile
    h->ring_maps.resize(2 * L);
    const size_t layer_bytes = Bm * d.Hkv * d.W * d.dh * es;
    const long long rows = (long long)Bm * d.Hkv * d.W;
    for (size_t l = 0; l < L && s == HF_OK; ++l) {
      e = hf::make_map(&h->ring_maps[2 * l], bptr(h->ring_k, l * layer_bytes), rows, d.dh, d.dh,
                       hf::attn_tile_rows(d));
      if (e == cudaSuccess)
        e = hf::make_map(&h->ring_maps[2 * l + 1], bptr(h->ring_v, l * layer_bytes), rows, d.dh,
                         d.dh, hf::attn_tile_rows(d));
      if (e != cudaSuccess) s = cuda_fail(h, e, "ring tensor maps");
    }
    if (s == HF_OK && hf::mem_tc_ok(d)) {
      h->state_maps.resize(L);
      const size_t sl_bytes = Bm * d.Hm * d.P * d.N * 4;
      for (size_t l = 0; l < L && s == HF_OK; ++l) {
        e = hf::make_map_f32(&h->state_maps[l], bptr(h->state, l * sl_bytes),
                             (long long)Bm * d.Hm * d.P, d.N, d.P);
        if (e != cudaSuccess) s = cuda_fail(h, e, "state tensor maps");
      }
    }
  }
  if (s == HF_OK) {
    e = hf::configure_attn_cluster(h->d);
    if (e == cudaSuccess && h->cfg.dtype == HF_BF16) e = hf::configure_tc();
    if (e == cudaSuccess && h->cfg.dtype == HF_BF16) e = hf::configure_tc_persistent(h->num_sms);
    if (e == cudaSuccess && h->cfg.dtype == HF_BF16) e = hf::configure_gemm_sk();
    if (e == cudaSuccess && h->cfg.dtype == HF_BF16) e = hf::configure_gemm_tm();
    if (e == cudaSuccess) e = hf::configure_commit_state(h->d);
    if (e != cudaSuccess) s = cuda_fail(h, e, "kernel set-up");
  }
  if (s == HF_OK) {
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) s = cuda_fail(h, e, "cudaDeviceSynchronize");
  }
  if (s != HF_OK) {
    g_create_error = h->msg;
    free_all(h);
    delete h;
    return s;
  }
  *out = h;
  return HF_OK;
}

void hf_destroy(hf_handle* h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
}

// The 4-bit side of a layer upload: codes / parameters in the per-call-site
// row order of the bf16 weights (rows = output features, K = inputs).
struct Q4Site {
  std::vector<uint8_t> codes;  // [M][K]
  std::vector<uint32_t> prm;   // [M][K/128]: scale bits | zero << 16
  long long M = 0, K = 0;
  void init(long long m, long long k) {
    M = m;
    K = k;
    codes.assign((size_t)m * k, 0);
    prm.assign((size_t)m * (k / 128), 0);
  }
  // matrix [in, outn] (q4 form) into rows row0.. and input columns col0..
  void put(const hf_q4_matrix& q, size_t row0, size_t col0, size_t in, size_t outn) {
    for (size_t i = 0; i < in; ++i)
      for (size_t o = 0; o < outn; ++o) codes[(row0 + o) * K + col0 + i] = q.codes[i * outn + o];
    for (size_t g = 0; g < in / 128; ++g)
      for (size_t o = 0; o < outn; ++o)
        prm[(row0 + o) * (K / 128) + col0 / 128 + g] =
            (uint32_t)q.scales[g * outn + o] | ((uint32_t)q.zeros[g * outn + o] << 16);
  }
};
struct Q4Layer {
  Q4Site draft, commit, out;
};

static hf_status upload_layer(hf_handle* h, int32_t layer, const hf_layer_weights* w,
                              const hf_layer_weights_q4* q, const void* w_z = nullptr);

hf_status hf_set_weights(hf_handle* h, int32_t layer, const hf_layer_weights* w) {
  if (!h) return HF_EINVAL;
  if (h->q4) return fail(h, HF_EINVAL, "weight_bits = 4: set the weights with hf_set_weights_q4");
  if (h->d.blk) return fail(h, HF_EINVAL, "full block: set the weights with hf_set_block_weights");
  return upload_layer(h, layer, w, nullptr);
}

// Transpose a host [in, out] matrix (element size es) into [out][in] rows.
static std::vector<char> transposed(const void* src, size_t in, size_t outn, size_t es) {
  std::vector<char> t(in * outn * es);
  const char* s = static_cast<const char*>(src);
  for (size_t i = 0; i < in; ++i)
    for (size_t o = 0; o < outn; ++o) std::memcpy(&t[(o * in + i) * es], s + (i * outn + o) * es, es);
  return t;
}

// Copy a [rows][K] weight (model dtype) and, for bf16 handles, its tiles.
static hf_status put_weight(hf_handle* h, const std::vector<char>& w, long long rows, long long K,
                            void* dst, void* tiles) {
  HF_CUDA(h, cudaMemcpy(dst, w.data(), w.size(), cudaMemcpyHostToDevice));
  if (tiles) {
    std::vector<uint16_t> t(hf::tiled_bytes(rows, K) / 2);
    hf::tile_weights(reinterpret_cast<const uint16_t*>(w.data()), rows, K, t.data());
    HF_CUDA(h, cudaMemcpy(tiles, t.data(), t.size() * 2, cudaMemcpyHostToDevice));
  }
  return HF_OK;
}

hf_status hf_set_block_weights(hf_handle* h, int32_t layer, const hf_layer_weights* w,
                               const hf_block_weights* bw) {
  if (!h) return HF_EINVAL;
  const Dims& d = h->d;
  if (!d.blk) return fail(h, HF_EINVAL, "hf_set_block_weights needs a full-block handle");
  if (!w || !bw || layer < 0 || layer >= d.L) return fail(h, HF_EINVAL, "bad layer or weights");
  const void* ptrs[] = {bw->g_mix, bw->g_mlp, bw->w_z, bw->d_skip, bw->conv_w,
                        bw->conv_b, bw->w_gate, bw->w_up, bw->w_down};
  for (const void* p : ptrs)
    if (!p) return fail(h, HF_EINVAL, "a block weight pointer is NULL");
  hf_status s = upload_layer(h, layer, w, nullptr, bw->w_z);
  if (s != HF_OK) return s;
  const size_t es = h->esz, D = d.D, F = d.F, C = d.dinner + d.N;
  HF_CUDA(h, cudaMemcpy(h->g_mix + (size_t)layer * D, bw->g_mix, D * 4, cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(h->g_mlp + (size_t)layer * D, bw->g_mlp, D * 4, cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(h->d_skip + (size_t)layer * d.Hm, bw->d_skip, d.Hm * 4, cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(h->conv_w + (size_t)layer * C * 4, bw->conv_w, C * 4 * 4, cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(h->conv_b + (size_t)layer * C, bw->conv_b, C * 4, cudaMemcpyHostToDevice));
  // [W_gate^T ; W_up^T] rows, and W_down^T
  std::vector<char> up = transposed(bw->w_gate, D, F, es);
  const std::vector<char> u2 = transposed(bw->w_up, D, F, es);
  up.insert(up.end(), u2.begin(), u2.end());
  const std::vector<char> down = transposed(bw->w_down, F, D, es);
  if ((s = put_weight(h, up, 2 * F, D, bptr(h->w_up, layer * up.size()),
                      h->wt_up ? bptr(h->wt_up, layer * h->wt_up_l) : nullptr)) != HF_OK)
    return s;
  if ((s = put_weight(h, down, D, F, bptr(h->w_down, layer * down.size()),
                      h->wt_down ? bptr(h->wt_down, layer * h->wt_down_l) : nullptr)) != HF_OK)
    return s;
  HF_CUDA(h, cudaDeviceSynchronize());
  return HF_OK;
}

hf_status hf_set_head_weights(hf_handle* h, const float* g_final, const void* w_lm) {
  if (!h) return HF_EINVAL;
  const Dims& d = h->d;
  if (!d.blk) return fail(h, HF_EINVAL, "hf_set_head_weights needs a full-block handle");
  if (!g_final || !w_lm) return fail(h, HF_EINVAL, "a head weight pointer is NULL");
  HF_CUDA(h, cudaSetDevice(h->device));
  HF_CUDA(h, cudaMemcpy(h->g_final, g_final, (size_t)d.D * 4, cudaMemcpyHostToDevice));
  const std::vector<char> lm = transposed(w_lm, d.D, d.V, h->esz);
  hf_status s = put_weight(h, lm, d.V, d.D, h->w_lm, h->wt_lm);
  if (s != HF_OK) return s;
  HF_CUDA(h, cudaDeviceSynchronize());
  h->head_set = 1;
  return HF_OK;
}

// bf16 bits, round to nearest even (finite inputs)
static uint16_t to_bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

hf_status hf_set_weights_q4(hf_handle* h, int32_t layer, const hf_layer_weights_q4* q) {
  if (!h) return HF_EINVAL;
  if (!h->q4) return fail(h, HF_EINVAL, "hf_set_weights_q4 needs a handle with weight_bits = 4");
  if (!q || layer < 0 || layer >= h->d.L) return fail(h, HF_EINVAL, "bad layer or weights");
  const Dims& d = h->d;
  const hf_q4_matrix* mats[] = {&q->w_q, &q->w_k, &q->w_v, &q->w_o, &q->w_x, &q->w_B,
                                &q->w_C, &q->w_dt, &q->w_mo, &q->w_beta};
  const size_t ins[] = {(size_t)d.D, (size_t)d.D, (size_t)d.D, (size_t)d.QD, (size_t)d.D,
                        (size_t)d.D, (size_t)d.D, (size_t)d.D, (size_t)d.dinner, (size_t)d.D};
  const size_t outs[] = {(size_t)d.QD, (size_t)d.KVD, (size_t)d.KVD, (size_t)d.D, (size_t)d.dinner,
                         (size_t)d.N, (size_t)d.N, (size_t)d.Hm, (size_t)d.D, (size_t)d.Hm};
  const int nm = d.gdn ? 10 : 9;
  if (!q->dt_bias || !q->A_log) return fail(h, HF_EINVAL, "a weight pointer is NULL");
  // dequantise on the host (w = s * (code - zero), one rounding to bf16: the
  // product of a bf16 scale and a 4-bit integer is exact in fp32)
  std::vector<std::vector<uint16_t>> deq(nm);
  for (int m = 0; m < nm; ++m) {
    const hf_q4_matrix& x = *mats[m];
    if (!x.codes || !x.scales || !x.zeros) return fail(h, HF_EINVAL, "a weight pointer is NULL");
    const size_t in = ins[m], on = outs[m];
    deq[m].resize(in * on);
    for (size_t i = 0; i < in; ++i)
      for (size_t o = 0; o < on; ++o) {
        const uint8_t c = x.codes[i * on + o], z = x.zeros[(i / 128) * on + o];
        if (c > 15 || z > 15) return fail(h, HF_EINVAL, "4-bit codes and zeros must be 0..15");
        uint32_t sb = (uint32_t)x.scales[(i / 128) * on + o] << 16;
        float sc;
        std::memcpy(&sc, &sb, 4);
        deq[m][i * on + o] = to_bf16_bits(sc * ((float)c - (float)z));
      }
  }
  hf_layer_weights wb{};
  wb.w_q = deq[0].data();
  wb.w_k = deq[1].data();
  wb.w_v = deq[2].data();
  wb.w_o = deq[3].data();
  wb.w_x = deq[4].data();
  wb.w_B = deq[5].data();
  wb.w_C = deq[6].data();
  wb.w_dt = deq[7].data();
  wb.w_mo = deq[8].data();
  wb.w_beta = d.gdn ? deq[9].data() : nullptr;
  wb.dt_bias = q->dt_bias;
  wb.A_log = q->A_log;
  return upload_layer(h, layer, &wb, q);
}

static hf_status upload_layer(hf_handle* h, int32_t layer, const hf_layer_weights* w,
                              const hf_layer_weights_q4* q, const void* w_z) {
  if (!w || layer < 0 || layer >= h->d.L) return fail(h, HF_EINVAL, "bad layer or weights");
  const void* ptrs[] = {w->w_q, w->w_k, w->w_v, w->w_o, w->w_x, w->w_B, w->w_C, w->w_dt, w->w_mo,
                        w->dt_bias, w->A_log};
  for (const void* p : ptrs)
    if (!p) return fail(h, HF_EINVAL, "a weight pointer is NULL");
  if (h->d.gdn && !w->w_beta) return fail(h, HF_EINVAL, "the gated-delta memory needs w_beta");
  HF_CUDA(h, cudaSetDevice(h->device));
  const Dims& d = h->d;
  const size_t es = h->esz, D = d.D;
  // Transpose a host [in, out] matrix into rows [out][in] of dst (row length ld).
  auto put_t = [&](std::vector<char>& dst, size_t row0, size_t ld, const void* src, size_t in,
                   size_t outn) {
    const char* s = static_cast<const char*>(src);
    for (size_t i = 0; i < in; ++i)
      for (size_t o = 0; o < outn; ++o)
        std::memcpy(&dst[((row0 + o) * ld + i) * es], s + (i * outn + o) * es, es);
  };
  std::vector<char> wd((size_t)d.Nd * D * es), wc((size_t)d.Nc * D * es), wo((size_t)D * d.Nz * es);
  put_t(wd, 0, D, w->w_q, D, d.QD);
  put_t(wd, d.QD, D, w->w_k, D, d.KVD);
  put_t(wd, d.QD + d.KVD, D, w->w_v, D, d.KVD);
  put_t(wd, d.QD + 2 * d.KVD, D, w->w_C, D, d.N);
  if (d.blk) {  // full block: x_s and z_s of the memory read's skip and gate
    put_t(wd, d.QD + 2 * d.KVD + d.N, D, w->w_x, D, d.dinner);
    put_t(wd, d.QD + 2 * d.KVD + d.N + d.dinner, D, w_z, D, d.dinner);
  }
  put_t(wc, 0, D, w->w_k, D, d.KVD);
  put_t(wc, d.KVD, D, w->w_v, D, d.KVD);
  put_t(wc, 2 * d.KVD, D, w->w_x, D, d.dinner);
  put_t(wc, 2 * d.KVD + d.dinner, D, w->w_B, D, d.N);
  put_t(wc, 2 * d.KVD + d.dinner + d.N, D, w->w_dt, D, d.Hm);
  if (d.gdn) put_t(wc, 2 * d.KVD + d.dinner + d.N + d.Hm, D, w->w_beta, D, d.Hm);
  // W_out^T: row c = [W_o[:, c] | W_mo[:, c]]
  {
    const char* so = static_cast<const char*>(w->w_o);
    const char* sm = static_cast<const char*>(w->w_mo);
    for (size_t k = 0; k < (size_t)d.QD; ++k)
      for (size_t c = 0; c < D; ++c) std::memcpy(&wo[(c * d.Nz + k) * es], so + (k * D + c) * es, es);
    for (size_t k = 0; k < (size_t)d.dinner; ++k)
      for (size_t c = 0; c < D; ++c)
        std::memcpy(&wo[(c * d.Nz + d.QD + k) * es], sm + (k * D + c) * es, es);
  }
  HF_CUDA(h, cudaMemcpy(bptr(h->w_draft, (size_t)layer * wd.size()), wd.data(), wd.size(), cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(bptr(h->w_commit, (size_t)layer * wc.size()), wc.data(), wc.size(), cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(bptr(h->w_out, (size_t)layer * wo.size()), wo.data(), wo.size(), cudaMemcpyHostToDevice));
  if (q) {  // 4-bit tiles of the three call sites, rows as in wd / wc / wo
    Q4Layer ql;
    ql.draft.init(d.Nd, D);
    ql.draft.put(q->w_q, 0, 0, D, d.QD);
    ql.draft.put(q->w_k, d.QD, 0, D, d.KVD);
    ql.draft.put(q->w_v, d.QD + d.KVD, 0, D, d.KVD);
    ql.draft.put(q->w_C, d.QD + 2 * d.KVD, 0, D, d.N);
    ql.commit.init(d.Nc, D);
    ql.commit.put(q->w_k, 0, 0, D, d.KVD);
    ql.commit.put(q->w_v, d.KVD, 0, D, d.KVD);
    ql.commit.put(q->w_x, 2 * d.KVD, 0, D, d.dinner);
    ql.commit.put(q->w_B, 2 * d.KVD + d.dinner, 0, D, d.N);
    ql.commit.put(q->w_dt, 2 * d.KVD + d.dinner + d.N, 0, D, d.Hm);
    if (d.gdn) ql.commit.put(q->w_beta, 2 * d.KVD + d.dinner + d.N + d.Hm, 0, D, d.Hm);
    ql.out.init(D, d.Nz);
    ql.out.put(q->w_o, 0, 0, d.QD, D);
    ql.out.put(q->w_mo, 0, d.QD, d.dinner, D);
    std::vector<uint8_t> t(std::max({h->wt_draft_l, h->wt_commit_l, h->wt_out_l}));
    struct {
      Q4Site* site;
      long long rows;
      void* dst;
      size_t bytes;
    } jobs[] = {{&ql.draft, d.Nd, h->wt_draft, h->wt_draft_l},
                {&ql.commit, h->nc_pad, h->wt_commit, h->wt_commit_l},
                {&ql.out, D, h->wt_out, h->wt_out_l}};
    for (auto& j : jobs) {
      // rows past the site's (commit padding) are zero codes and parameters
      j.site->codes.resize((size_t)j.rows * j.site->K, 0);
      j.site->prm.resize((size_t)j.rows * (j.site->K / 128), 0);
      hf::tile_weights_q4(j.site->codes.data(), j.site->prm.data(), j.rows, j.site->K, t.data());
      HF_CUDA(h, cudaMemcpy(bptr(j.dst, (size_t)layer * j.bytes), t.data(), j.bytes,
                            cudaMemcpyHostToDevice));
    }
  } else if (h->cfg.dtype == HF_BF16) {
    std::vector<uint16_t> t(std::max({h->wt_draft_l, h->wt_commit_l, h->wt_out_l}) / 2);
    hf::tile_weights(reinterpret_cast<const uint16_t*>(wd.data()), d.Nd, D, t.data());
    HF_CUDA(h, cudaMemcpy(bptr(h->wt_draft, (size_t)layer * h->wt_draft_l), t.data(), h->wt_draft_l,
                          cudaMemcpyHostToDevice));
    hf::tile_weights(reinterpret_cast<const uint16_t*>(wc.data()), d.Nc, D, t.data());
    HF_CUDA(h, cudaMemcpy(bptr(h->wt_commit, (size_t)layer * h->wt_commit_l), t.data(),
                          h->wt_commit_l, cudaMemcpyHostToDevice));
    hf::tile_weights(reinterpret_cast<const uint16_t*>(wo.data()), D, d.Nz, t.data());
    HF_CUDA(h, cudaMemcpy(bptr(h->wt_out, (size_t)layer * h->wt_out_l), t.data(), h->wt_out_l,
                          cudaMemcpyHostToDevice));
  }
  HF_CUDA(h, cudaMemcpy(h->dt_bias + (size_t)layer * d.Hm, w->dt_bias, d.Hm * 4, cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaMemcpy(h->A_log + (size_t)layer * d.Hm, w->A_log, d.Hm * 4, cudaMemcpyHostToDevice));
  HF_CUDA(h, cudaDeviceSynchronize());
  return HF_OK;
}

namespace {

// Attention launch: what it may read before its dependency wait (ring K/V,
// positions and states, slot projections).
constexpr int kEarlyRing = 1, kEarlyState = 2, kEarlyProj = 4;
// hf_round folds the first layer's memory read into the state update once a
// layer's states are at least this large (below, the read runs beside the
// attention, off the round's critical path).
constexpr size_t kFuseMemBytes = 16u << 20;

// Slot projections of draft layer l (rows of X) into h->proj. With the
// tensor-core attention the GEMM signals its dependents only after its own
// dependency wait, so that the attention launch may read the ring, positions
// and state (final by then) before its wait.
hf_status draft_proj(hf_handle* h, int l, const void* X, int batch, int late, cudaStream_t st) {
  const Dims& d = h->d;
  Epi e1 = epi_base(h);
  e1.kind = hf::EPI_F32;
  e1.out = h->proj;
  e1.ld = d.Nd;
  return gemm(h, HF_K_DRAFT_PROJ, X, d.D, bptr(h->w_draft, (size_t)l * d.Nd * d.D * h->esz), d.D,
              batch * d.S, d.Nd, d.D, e1, st,
              h->wt_draft ? bptr(h->wt_draft, (size_t)l * h->wt_draft_l) : nullptr, late);
}

// The rest of draft layer l once its slot projections are in h->proj:
// attention (+ memory read unless with_mem = 0) into h->mix, then the
// output projection with the residual X into Y.
hf_status draft_rest(hf_handle* h, int l, const void* X, void* Y, int batch, int early,
                     int with_mem, cudaStream_t st) {
  const Dims& d = h->d;
  const size_t es = h->esz;
  const size_t ring_ls = (size_t)d.Bmax * d.Hkv * d.W * d.dh * es;
  const size_t state_ls = (size_t)d.Bmax * d.Hm * d.P * d.N;
  {
    Scope sc(h, HF_K_ATTN_MEM, st);
    const CUtensorMap* mk = h->ring_maps.empty() ? nullptr : &h->ring_maps[2 * l];
    const CUtensorMap* mv = h->ring_maps.empty() ? nullptr : &h->ring_maps[2 * l + 1];
    const CUtensorMap* ms = h->state_maps.empty() ? nullptr : &h->state_maps[l];
    cudaError_t e = hf::launch_attn_cluster(h->cfg.dtype, d, batch, h->proj,
                                            bptr(h->ring_k, l * ring_ls),
                                            bptr(h->ring_v, l * ring_ls), h->pos,
                                            h->state + l * state_ls, h->mix, mk, mv, ms, h->err,
                                            h->num_sms, early, with_mem, st, &sc.count);
    if (e != cudaSuccess) return cuda_fail(h, e, "attention launch");
  }
  Epi e2 = epi_base(h);
  e2.kind = hf::EPI_RESID;
  e2.resid = X;
  e2.out_t = Y;
  e2.ld = d.D;
  return gemm(h, HF_K_OUT_PROJ, h->mix, d.Nz, bptr(h->w_out, (size_t)l * d.D * d.Nz * es), d.Nz,
              batch * d.S, d.D, d.Nz, e2, st,
              h->wt_out ? bptr(h->wt_out, (size_t)l * h->wt_out_l) : nullptr);
}

// One layer of the full drafter block: X -> Y (rows batch*S).
//   a = RMSNorm(X; g_mix) -> [Q | K_s | V_s | C_s | x_s | z_s] = a W (fp32)
//   -> RoPE of Q, K_s at pos + s -> attention O and memory read y
//   -> y <- (y + D x_s) silu(z_s) -> X1 = X + [O | y] W_out
//   -> n = RMSNorm(X1; g_mlp) -> [g | u] = n [W_gate | W_up] -> act = silu(g) u
//   -> Y = X1 + act W_down
hf_status draft_block_layer(hf_handle* h, int l, const void* X, void* Y, int batch,
                            cudaStream_t st) {
  const Dims& d = h->d;
  const size_t es = h->esz;
  const int rows = batch * d.S, dt = h->cfg.dtype;
  cudaError_t e;
  {
    Scope sc(h, HF_K_OTHER, st);
    e = hf::launch_rms_norm(dt, X, h->g_mix + (size_t)l * d.D, h->anorm, rows, d.D, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "rms_norm launch");
  }
  hf_status s = draft_proj(h, l, h->anorm, batch, 0, st);
  if (s != HF_OK) return s;
  {
    Scope sc(h, HF_K_OTHER, st);
    e = hf::launch_rope_slots(d, rows, h->proj, h->pos, h->rope_inv, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "rope launch");
  }
  const size_t ring_ls = (size_t)d.Bmax * d.Hkv * d.W * d.dh * es;
  const size_t state_ls = (size_t)d.Bmax * d.Hm * d.P * d.N;
  {
    Scope sc(h, HF_K_ATTN_MEM, st);
    const CUtensorMap* mk = h->ring_maps.empty() ? nullptr : &h->ring_maps[2 * l];
    const CUtensorMap* mv = h->ring_maps.empty() ? nullptr : &h->ring_maps[2 * l + 1];
    const CUtensorMap* ms = h->state_maps.empty() ? nullptr : &h->state_maps[l];
    e = hf::launch_attn_cluster(dt, d, batch, h->proj, bptr(h->ring_k, l * ring_ls),
                                bptr(h->ring_v, l * ring_ls), h->pos, h->state + l * state_ls,
                                h->mix, mk, mv, ms, h->err, h->num_sms, 0, 1, st, &sc.count);
    if (e != cudaSuccess) return cuda_fail(h, e, "attention launch");
  }
  {
    Scope sc(h, HF_K_OTHER, st);
    e = hf::launch_gate_skip(dt, d, rows, h->mix, h->proj, h->d_skip + (size_t)l * d.Hm, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "gate launch");
  }
  Epi e2 = epi_base(h);
  e2.kind = hf::EPI_RESID;
  e2.resid = X;
  e2.out_t = h->x1;
  e2.ld = d.D;
  s = gemm(h, HF_K_OUT_PROJ, h->mix, d.Nz, bptr(h->w_out, (size_t)l * d.D * d.Nz * es), d.Nz,
           rows, d.D, d.Nz, e2, st, h->wt_out ? bptr(h->wt_out, (size_t)l * h->wt_out_l) : nullptr);
  if (s != HF_OK) return s;
  {
    Scope sc(h, HF_K_OTHER, st);
    e = hf::launch_rms_norm(dt, h->x1, h->g_mlp + (size_t)l * d.D, h->anorm, rows, d.D, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "rms_norm launch");
  }
  Epi eu = epi_base(h);
  eu.kind = hf::EPI_F32;
  eu.out = h->mlp_h;
  eu.ld = 2 * d.F;
  s = gemm(h, HF_K_MLP, h->anorm, d.D, bptr(h->w_up, (size_t)l * 2 * d.F * d.D * es), d.D, rows,
           2 * d.F, d.D, eu, st, h->wt_up ? bptr(h->wt_up, (size_t)l * h->wt_up_l) : nullptr);
  if (s != HF_OK) return s;
  {
    Scope sc(h, HF_K_MLP, st);
    e = hf::launch_swiglu(dt, rows, d.F, h->mlp_h, h->act, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "swiglu launch");
  }
  Epi ed = epi_base(h);
  ed.kind = hf::EPI_RESID;
  ed.resid = h->x1;
  ed.out_t = Y;
  ed.ld = d.D;
  return gemm(h, HF_K_MLP, h->act, d.F, bptr(h->w_down, (size_t)l * d.D * d.F * es), d.F, rows,
              d.D, d.F, ed, st, h->wt_down ? bptr(h->wt_down, (size_t)l * h->wt_down_l) : nullptr);
}

// The LM head of a block handle: logits = RMSNorm(X; g_final) W_lm, tokens =
// row argmax (ties to the lowest id).
hf_status draft_head(hf_handle* h, const void* X, int32_t* tokens, int batch, cudaStream_t st) {
  const Dims& d = h->d;
  const int rows = batch * d.S;
  cudaError_t e;
  {
    Scope sc(h, HF_K_OTHER, st);
    e = hf::launch_rms_norm(h->cfg.dtype, X, h->g_final, h->anorm, rows, d.D, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "rms_norm launch");
  }
  Epi el = epi_base(h);
  el.kind = hf::EPI_F32;
  el.out = h->logits;
  el.ld = d.V;
  hf_status s = gemm(h, HF_K_HEAD, h->anorm, d.D, h->w_lm, d.D, rows, d.V, d.D, el, st, h->wt_lm);
  if (s != HF_OK) return s;
  Scope sc(h, HF_K_HEAD, st);
  e = hf::launch_argmax(rows, d.V, h->logits, tokens, st);
  sc.count = 1;
  if (e != cudaSuccess) return cuda_fail(h, e, "argmax launch");
  return HF_OK;
}

// Commit-projection epilogue: of the batch*(S+1) rows of every layer only
// rows t < n_b are kept (ring append at pos_b + t; x, B, dt into xbd).
Epi commit_epi(const hf_handle* h, const int32_t* n_accepted) {
  const Dims& d = h->d;
  Epi ep = epi_base(h);
  ep.kind = hf::EPI_SSM_KV;
  ep.layer0 = 0;
  ep.cols_per_layer = d.Nc;
  ep.col_off = 0;
  ep.n_acc = n_accepted;
  ep.pos = h->pos;
  ep.xbd = h->xbd;
  ep.xbd_layer_stride = h->xbd_ls;
  ep.pos_snap = h->pos_snap;  // memory horizon M > 1 only (else NULL)
  if (h->wt_commit) {  // pre-tiled: rows padded per layer to nc_pad, padding skipped
    ep.cols_per_layer = h->nc_pad;
    ep.cols_valid = d.Nc;
  }
  return ep;
}

// early: the commit projection signalled its dependents after its wait;
// late: the next launch reads the ring before its own wait.
// The commit epilogue over the plain (unpadded) commit weights.
Epi plain_commit_epi(const hf_handle* h, const int32_t* n_accepted) {
  Epi ep = commit_epi(h, n_accepted);
  ep.cols_per_layer = h->d.Nc;
  ep.cols_valid = 0;
  return ep;
}

hf_status commit_state(hf_handle* h, const int32_t* n_accepted, int batch, const float* memC,
                       int early, int late, cudaStream_t st) {
  const Dims& d = h->d;
  Scope sc(h, HF_K_COMMIT_STATE, st);
  const hf::MemRing mr{h->mem_x, h->mem_b, h->mem_dt, h->pos_snap};
  cudaError_t e = hf::launch_commit_state(h->cfg.dtype, d, batch, n_accepted, h->xbd, h->xbd_ls,
                                          h->A_log, h->state, h->pos, h->offsets, h->tags, h->err,
                                          memC, h->mix, early, late, h->num_sms, mr, st);
  sc.count = 1;
  if (e != cudaSuccess) return cuda_fail(h, e, "commit state launch");
  return HF_OK;
}

hf_status check_draft_args(hf_handle* h, const void* slot_emb, void* out, int32_t batch) {
  if (!slot_emb || !out) return fail(h, HF_EINVAL, "NULL buffer");
  if (batch < 0 || batch > h->d.Bmax) return fail(h, HF_EINVAL, "batch out of range");
  if (slot_emb == out) return fail(h, HF_EINVAL, "out may not alias slot_emb");
  if (reinterpret_cast<uintptr_t>(slot_emb) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(h, HF_EINVAL, "slot_emb and out must be 16-byte aligned");
  return HF_OK;
}

hf_status check_commit_args(hf_handle* h, const void* feats, const int32_t* n_accepted,
                            int32_t batch) {
  if (!feats || !n_accepted) return fail(h, HF_EINVAL, "NULL buffer");
  if (reinterpret_cast<uintptr_t>(feats) % 16) return fail(h, HF_EINVAL, "feats must be 16-byte aligned");
  if (batch < 0 || batch > h->d.Bmax) return fail(h, HF_EINVAL, "batch out of range");
  return HF_OK;
}

}  // namespace

hf_status hf_draft(hf_handle* h, const void* slot_emb, void* out, int32_t batch, void* stream) {
  if (!h) return HF_EINVAL;
  hf_status s = check_draft_args(h, slot_emb, out, batch);
  if (s != HF_OK || batch == 0) return s;
  HF_CUDA(h, ensure_device(h));
  cudaStream_t st = (cudaStream_t)stream;
  const Dims& d = h->d;
  const bool tc = !h->ring_maps.empty();
  for (int l = 0; l < d.L; ++l) {
    const void* X = l == 0 ? slot_emb : h->xbuf[(l - 1) % 2];
    void* Y = l == d.L - 1 ? out : h->xbuf[l % 2];
    if (d.blk) {
      if ((s = draft_block_layer(h, l, X, Y, batch, st)) != HF_OK) return s;
      continue;
    }
    if ((s = draft_proj(h, l, X, batch, tc, st)) != HF_OK) return s;
    if ((s = draft_rest(h, l, X, Y, batch, tc ? kEarlyRing | kEarlyState : 0, 1, st)) != HF_OK)
      return s;
  }
  return HF_OK;
}

hf_status hf_draft_tokens(hf_handle* h, const void* slot_emb, void* out, int32_t* tokens,
                          int32_t batch, void* stream) {
  if (!h) return HF_EINVAL;
  if (!h->d.blk) return fail(h, HF_EINVAL, "hf_draft_tokens needs a full-block handle");
  if (!h->head_set) return fail(h, HF_EINVAL, "hf_draft_tokens: set the head weights first");
  if (!tokens) return fail(h, HF_EINVAL, "NULL buffer");
  hf_status s = hf_draft(h, slot_emb, out, batch, stream);
  if (s != HF_OK || batch == 0) return s;
  return draft_head(h, out, tokens, batch, (cudaStream_t)stream);
}

hf_status hf_commit(hf_handle* h, const void* feats, const int32_t* n_accepted, int32_t batch,
                    void* stream) {
  if (!h) return HF_EINVAL;
  hf_status s = check_commit_args(h, feats, n_accepted, batch);
  if (s != HF_OK || batch == 0) return s;
  HF_CUDA(h, ensure_device(h));
  cudaStream_t st = (cudaStream_t)stream;
  const Dims& d = h->d;
  // Projections of all batch*(S+1) rows of all layers in one GEMM.
  const Epi ep = commit_epi(h, n_accepted);
  const int rows = batch * (d.S + 1);
  const int late = h->cfg.dtype == HF_BF16 ? 1 : 0;  // the tensor-core GEMM can signal late
  // the tiled commit weights are one matrix per layer, stacked; wide batches
  // run token-major over the plain weights
  const bool tiled = h->wt_commit && rows <= 32;
  s = gemm(h, HF_K_COMMIT_PROJ, feats, d.D, h->w_commit, d.D, rows,
           d.L * (tiled ? h->nc_pad : d.Nc), d.D, tiled ? ep : plain_commit_epi(h, n_accepted), st,
           tiled ? h->wt_commit : nullptr, late, h->nc_pad / 128);
  if (s != HF_OK) return s;
  if (d.blk) {
    // full block: rotate the appended keys at their positions, convolve the
    // accepted rows' x | B with the carried rows (in place, before the
    // state update reads them); signals its dependents after its own wait
    Scope sc(h, HF_K_COMMIT_STATE, st);
    cudaError_t e = hf::launch_commit_prep(h->cfg.dtype, d, batch, n_accepted, h->pos, h->ring_k,
                                           h->xbd, h->xbd_ls, h->conv_state, h->conv_w,
                                           h->conv_b, h->rope_inv, st);
    sc.count = 1;
    if (e != cudaSuccess) return cuda_fail(h, e, "commit prep launch");
    return commit_state(h, n_accepted, batch, nullptr, 1, 0, st);
  }
  return commit_state(h, n_accepted, batch, nullptr, late, 0, st);
}

hf_status hf_round(hf_handle* h, const void* feats, const int32_t* n_accepted,
                   const void* slot_emb, void* out, int32_t batch, void* stream) {
  if (!h) return HF_EINVAL;
  hf_status s = check_commit_args(h, feats, n_accepted, batch);
  if (s == HF_OK) s = check_draft_args(h, slot_emb, out, batch);
  if (s != HF_OK || batch == 0) return s;
  const bool fused = h->cfg.dtype == HF_BF16 && h->wt_commit && h->wt_draft &&
                     !h->ring_maps.empty() && !h->d.blk;
  if (!fused) {
    s = hf_commit(h, feats, n_accepted, batch, stream);
    return s != HF_OK ? s : hf_draft(h, slot_emb, out, batch, stream);
  }
  HF_CUDA(h, ensure_device(h));
  cudaStream_t st = (cudaStream_t)stream;
  const Dims& d = h->d;
  // 1. commit projection (all layers) and the layer-0 slot projection in one
  //    grouped launch: both stream their weights at once
  {
    const Epi ec = commit_epi(h, n_accepted);
    Epi e1 = epi_base(h);
    e1.kind = hf::EPI_F32;
    e1.out = h->proj;
    e1.ld = d.Nd;
    const int M0 = d.L * h->nc_pad, N0 = batch * (d.S + 1), N1 = batch * d.S;
    const int splits =
        hf::tc_pick_splits((M0 + 127) / 128 * 128 + d.Nd, std::max(N0, N1), d.D, h->q4);
    Scope sc(h, HF_K_ROUND_PROJ, st);
    const bool tm = std::max(N0, N1) > 32;  // wide batch: token-major over the plain weights
    const bool sk = !tm && !h->q4 && (M0 + 127) / 128 + (d.Nd + 127) / 128 > h->num_sms;
    // wide batch with a tile per SM in the commit product alone: the commit
    // projection on the persistent GEMM, then the slot projection (split-K
    // clusters), which signals its dependents after its own wait
    const bool two_launch = tm && (long long)((N0 + 127) / 128) * ((d.L * d.Nc + 255) / 256) >= h->num_sms;
    if (two_launch) {
      cudaError_t e = hf::launch_gemm_persistent(feats, d.D, N0, h->w_commit, d.D, d.L * d.Nc, d.D,
                                                 h->err, plain_commit_epi(h, n_accepted),
                                                 h->num_sms, st, &sc.count);
      if (e == cudaSuccess)
        // (slot embeddings and weights are inputs of the call: the slot
        // projection's main loop overlaps the commit projection's last tiles)
        e = hf::launch_gemm_tc(slot_emb, d.D, N1, h->w_draft, d.D, d.Nd, d.D, 0,
                               hf::tc_pick_splits(N1, d.Nd, d.D), h->err, e1, st, &sc.count, nullptr,
                               /*late_trigger=*/1, 0, 0, /*independent=*/1);
      if (e != cudaSuccess) return cuda_fail(h, e, "round projection launches");
    }
    cudaError_t e =
        two_launch ? cudaSuccess
        : tm  ? hf::launch_gemm_tm(feats, d.D, N0, h->w_commit, d.D, d.L * d.Nc,
                                 plain_commit_epi(h, n_accepted), slot_emb, d.D, N1, h->w_draft, d.D,
                                 d.Nd, e1, d.D, h->num_sms, h->skws, h->skws_floats, h->counters,
                                 h->n_counters, h->err, /*late_trigger=*/1, st, &sc.count)
        : sk  ? hf::launch_gemm_sk(h->wt_commit, M0, h->nc_pad / 128, feats, d.D, N0, ec, h->wt_draft,
                                 d.Nd, slot_emb, d.D, N1, e1, d.D, h->num_sms, h->skws,
                                 h->skws_floats, h->counters, h->n_counters, h->err,
                                 /*late_trigger=*/1, st, &sc.count)
            : hf::launch_gemm_tc_grouped(h->wt_commit, M0, h->nc_pad / 128, feats, d.D, N0, ec,
                                         h->wt_draft, d.Nd, slot_emb, d.D, N1, e1, d.D, splits,
                                         h->err, st, &sc.count, /*late_trigger=*/1, h->q4);
    if (e != cudaSuccess) return cuda_fail(h, e, "grouped projection launch");
  }
  // 2. state update; at large batch also the layer-0 memory read of the new
  //    state (the state is then read once per round); it starts early (the
  //    grouped projection signals late) and signals late itself, so that the
  //    attention may request its ring tiles before waiting
  const size_t state_layer_bytes = (size_t)batch * d.Hm * d.P * d.N * 4;
  const bool fuse_mem = hf::mem_tc_ok(d) && state_layer_bytes >= kFuseMemBytes;
  s = commit_state(h, n_accepted, batch, fuse_mem ? h->proj + d.QD + 2 * d.KVD : nullptr, 1, 1,
                   st);
  if (s != HF_OK) return s;
  // 3. layer 0: attention and output projection; later layers as in hf_draft
  for (int l = 0; l < d.L; ++l) {
    const void* X = l == 0 ? slot_emb : h->xbuf[(l - 1) % 2];
    void* Y = l == d.L - 1 ? out : h->xbuf[l % 2];
    if (l > 0 && (s = draft_proj(h, l, X, batch, 1, st)) != HF_OK) return s;
    const int with_mem = l > 0 || !fuse_mem;
    // layer 0 follows the state update, which signals late: the ring and the
    // slot projections (grouped launch) are final, the positions are not
    const int early = l > 0 ? kEarlyRing | kEarlyState : kEarlyRing | kEarlyProj;
    if ((s = draft_rest(h, l, X, Y, batch, early, with_mem, st)) != HF_OK) return s;
  }
  return HF_OK;
}

hf_status hf_prefill(hf_handle* h, const void* feats, const int32_t* lens, const int32_t* requests,
                     int32_t n_req, void* stream) {
  if (!h) return HF_EINVAL;
  const Dims& d = h->d;
  if (n_req < 0 || n_req > d.Bmax) return fail(h, HF_EINVAL, "n_req out of range");
  if (n_req == 0) return HF_OK;
  if (!lens) return fail(h, HF_EINVAL, "lens is NULL");
  std::vector<int32_t> reqs(n_req);
  std::vector<char> seen(d.Bmax, 0);
  long long total = 0, ring_rows = 0;
  for (int i = 0; i < n_req; ++i) {
    reqs[i] = requests ? requests[i] : i;
    if (reqs[i] < 0 || reqs[i] >= d.Bmax) return fail(h, HF_EINVAL, "request index out of range");
    if (seen[reqs[i]]) return fail(h, HF_EINVAL, "request named twice");
    seen[reqs[i]] = 1;
    if (lens[i] < 0) return fail(h, HF_EINVAL, "negative prefix length");
    total += lens[i];
    ring_rows += std::min<long long>(lens[i], d.W);
  }
  if (total > 0 && !feats) return fail(h, HF_EINVAL, "feats is NULL");
  if (reinterpret_cast<uintptr_t>(feats) % 16) return fail(h, HF_EINVAL, "feats must be 16-byte aligned");
  if (total > (long long)INT32_MAX) return fail(h, HF_EINVAL, "prefix too long");
  HF_CUDA(h, ensure_device(h));
  cudaStream_t st = (cudaStream_t)stream;
  const size_t es = h->esz;
  HF_CUDA(h, cudaMemcpyAsync(h->pf_lens, lens, n_req * 4, cudaMemcpyHostToDevice, st));
  HF_CUDA(h, cudaMemcpyAsync(h->pf_reqs, reqs.data(), n_req * 4, cudaMemcpyHostToDevice, st));
  Scope sc(h, HF_K_PREFILL, st);
  cudaError_t e = hf::launch_prefill_reset(d, n_req, h->pf_reqs, h->state, h->tags, h->pos, st);
  sc.count++;
  if (e != cudaSuccess) return cuda_fail(h, e, "prefill reset");
  if (d.blk) {  // the convolution starts from zero rows
    e = hf::launch_conv_reset(d, n_req, h->pf_reqs, h->conv_state, st);
    sc.count++;
    if (e != cudaSuccess) return cuda_fail(h, e, "prefill conv reset");
  }
  if (ring_rows > 0) {
    e = hf::launch_prefill_ring_prep(h->cfg.dtype, d, n_req, (int)ring_rows, h->pf_lens,
                                     h->pf_reqs, feats, h->row_req, h->row_pos, h->tags,
                                     h->packed, h->req_len, st);
    sc.count++;
    if (e != cudaSuccess) return cuda_fail(h, e, "prefill ring prep");
  }
  for (int l = 0; l < d.L; ++l) {
    const char* wl = bptr(h->w_commit, (size_t)l * d.Nc * d.D * es);
    if (ring_rows > 0) {
      Epi ek = epi_base(h);
      ek.kind = hf::EPI_SSM_KV;
      ek.layer0 = l;
      ek.cols_per_layer = 2 * d.KVD;
      ek.col_off = 0;
      ek.row_req = h->row_req;
      ek.row_pos = h->row_pos;
      e = gemm_launch(h, h->packed, d.D, wl, d.D, (int)ring_rows, 2 * d.KVD, d.D, ek, st,
                      &sc.count);
      if (e != cudaSuccess) return cuda_fail(h, e, "prefill kv gemm");
      if (d.blk) {  // keys rotated at their positions as they enter the window
        e = hf::launch_ring_rope(h->cfg.dtype, d, l, (int)ring_rows, h->row_req, h->row_pos,
                                 h->ring_k, h->rope_inv, st);
        sc.count++;
        if (e != cudaSuccess) return cuda_fail(h, e, "prefill ring rope");
      }
      if (d.Mr > 0) {
        // memory horizon M > 1: x, B, dt of each request's last M features
        // (among the window rows, M <= W) into the memory-input ring
        Epi em = epi_base(h);
        em.kind = hf::EPI_MEMRING;
        em.layer0 = l;
        em.row_req = h->row_req;
        em.row_pos = h->row_pos;
        em.req_len = h->req_len;
        em.mx = h->mem_x;
        em.mb = h->mem_b;
        em.mdt = h->mem_dt;
        e = gemm_launch(h, h->packed, d.D, wl + (size_t)2 * d.KVD * d.D * es, d.D, (int)ring_rows,
                        d.dinner + d.N + d.Hm, d.D, em, st, &sc.count);
        if (e != cudaSuccess) return cuda_fail(h, e, "prefill memory-input gemm");
      }
    }
    const long long Tseg = h->pf_tokens;
    if (d.gdn) {
      // Gated delta: per request and pass of at most Tseg tokens, x | B | dt |
      // beta of every token (the commit projection's columns and epilogue),
      // then the rule applied token by token (no chunked form here)
      const char* w_mem = wl + (size_t)2 * d.KVD * d.D * es;
      const int ncol = d.dinner + d.N + 2 * d.Hm;
      long long cu = 0;
      for (int i = 0; i < n_req; ++i) {
        const long long Li = lens[i];
        for (long long s0 = 0; s0 < Li; s0 += Tseg) {
          const int T = (int)std::min(Tseg, Li - s0);
          Epi eg = epi_base(h);
          eg.kind = hf::EPI_SSM_KV;  // rows of no request: every row kept, no ring columns
          eg.layer0 = l;
          eg.cols_per_layer = ncol;
          eg.col_off = 2 * d.KVD;
          eg.xbd = h->gdn_xs;
          eg.xbd_layer_stride = 0;
          e = tokens_gemm(h, bptr(feats, (size_t)(cu + s0) * d.D * es), T, w_mem, ncol, eg, st,
                          &sc.count);
          if (e != cudaSuccess) return cuda_fail(h, e, "prefill gated-delta projection");
          e = hf::launch_gdn_prefill(d, l, reqs[i], T, h->gdn_xs, h->A_log, h->state, st);
          sc.count++;
          if (e != cudaSuccess) return cuda_fail(h, e, "prefill gated-delta scan");
        }
        cu += Li;
      }
      continue;
    }
    // Memory fold, per request and segment of at most Tseg tokens:
    //   dt (transposed) -> chunked decay scan -> w*x, B (transposed, bf16/fp32)
    //   -> state = decay_seg * state + (w*x)^T B   (contraction over tokens)
    const int nx = d.dinner + d.N;
    const char* w_xb = wl + (size_t)2 * d.KVD * d.D * es;
    const char* w_dt = wl + (size_t)(2 * d.KVD + d.dinner + d.N) * d.D * es;
    long long cu = 0;
    for (int i = 0; i < n_req; ++i) {
      const long long Li = lens[i];
      float* st_b = h->state + (((size_t)l * d.Bmax + reqs[i]) * d.Hm * d.P) * d.N;
      // with a memory horizon M only the last M features are folded
      const long long first = d.Mh > 0 ? std::max(0LL, Li - d.Mh) : 0;
      for (long long s0 = first; s0 < Li; s0 += Tseg) {
        const int T = (int)std::min(Tseg, Li - s0);
        const void* fseg = bptr(feats, (size_t)(cu + s0) * d.D * es);
        Epi e1 = epi_base(h);
        e1.kind = hf::EPI_DT;
        e1.layer0 = l;
        e1.dtw = h->pf_dtw;
        e1.ldt = (int)Tseg;
        e = tokens_gemm(h, fseg, T, w_dt, d.Hm, e1, st, &sc.count);
        if (e != cudaSuccess) return cuda_fail(h, e, "prefill dt gemm");
        e = hf::launch_prefill_decay(d, l, T, (int)Tseg, h->cfg.chunk, h->pf_dtw, h->A_log,
                                     h->pf_decay, st);
        sc.count++;
        if (e != cudaSuccess) return cuda_fail(h, e, "prefill decay scan");
        if (d.blk) {
          // full block: pre-conv x | B rows, then the causal conv1d over the
          // pass (rows before it from the carried ones) writes w * x and B
          Epi eu = epi_base(h);
          eu.kind = hf::EPI_F32;
          eu.out = h->pf_u;
          eu.ld = nx;
          e = tokens_gemm(h, fseg, T, w_xb, nx, eu, st, &sc.count);
          if (e != cudaSuccess) return cuda_fail(h, e, "prefill x/B gemm");
          const size_t C = nx;
          float* hist = h->conv_state + ((size_t)l * d.Bmax + reqs[i]) * 3 * C;
          e = hf::launch_conv_prefill(h->cfg.dtype, d, T, (int)Tseg, h->pf_u, hist, h->pf_dtw,
                                      h->conv_w + (size_t)l * C * 4, h->conv_b + (size_t)l * C,
                                      h->pf_xsT, h->pf_bT, st);
          sc.count += 2;
          if (e != cudaSuccess) return cuda_fail(h, e, "prefill conv");
        } else {
          Epi e2 = epi_base(h);
          e2.kind = hf::EPI_XB;
          e2.dtw = h->pf_dtw;
          e2.ldt = (int)Tseg;
          e2.xsT = h->pf_xsT;
          e2.bT = h->pf_bT;
          e = tokens_gemm(h, fseg, T, w_xb, nx, e2, st, &sc.count);
          if (e != cudaSuccess) return cuda_fail(h, e, "prefill x/B gemm");
        }
        Epi e3 = epi_base(h);
        e3.kind = hf::EPI_STATE;
        e3.st = st_b;
        e3.seg_decay = h->pf_decay;
        if (h->cfg.dtype == HF_F32) {
          const int splits = pick_splits(h, d.dinner, d.N, T, 64, 64);
          e = hf::launch_gemm_fma(h->cfg.dtype, h->pf_xsT, (int)Tseg, h->pf_bT, (int)Tseg, d.dinner,
                                  d.N, T, splits, h->part, e3, st, &sc.count);
        } else {
          const int splits = hf::tc_pick_splits(d.dinner, d.N, T);
          e = hf::launch_gemm_tc(h->pf_xsT, Tseg, d.dinner, h->pf_bT, Tseg, d.N, T, 0, splits,
                                 h->err, e3, st, &sc.count);
        }
        if (e != cudaSuccess) return cuda_fail(h, e, "prefill contraction gemm");
      }
      cu += Li;
    }
  }
  e = hf::launch_prefill_finish(n_req, h->pf_lens, h->pf_reqs, h->pos, st);
  sc.count++;
  if (e != cudaSuccess) return cuda_fail(h, e, "prefill finish");
  return HF_OK;
}

hf_status hf_sync(hf_handle* h, void* stream) {
  if (!h) return HF_EINVAL;
  HF_CUDA(h, cudaSetDevice(h->device));
  HF_CUDA(h, cudaStreamSynchronize((cudaStream_t)stream));
  HF_CUDA(h, cudaGetLastError());
  int32_t word = 0;
  HF_CUDA(h, cudaMemcpy(&word, h->err, 4, cudaMemcpyDeviceToHost));
  if (word) {
    HF_CUDA(h, cudaMemset(h->err, 0, 4));
    std::string m;
    if (word & hf::ERR_BAD_ACCEPTED) m += "accepted count outside 0..block+1 (request left unchanged); ";
    if (word & hf::ERR_TIMEOUT) {
      m += "a bounded device wait gave up; ";
      // a launch that gave up may have left stream-K tickets raised
      HF_CUDA(h, cudaMemset(h->counters, 0, (size_t)h->n_counters * 4));
    }
    return fail(h, (word & hf::ERR_TIMEOUT) ? HF_ETIMEOUT : HF_EDEVICE, m);
  }
  return HF_OK;
}

hf_status hf_tensor_bytes(const hf_handle* h, int32_t which, size_t* bytes) {
  if (!h || !bytes) return HF_EINVAL;
  const Dims& d = h->d;
  const size_t L = d.L, Bm = d.Bmax;
  switch (which) {
    case HF_T_STATE: *bytes = L * Bm * d.Hm * d.P * d.N * 4; break;
    case HF_T_RING_K:
    case HF_T_RING_V: *bytes = L * Bm * d.Hkv * d.W * d.dh * h->esz; break;
    case HF_T_RING_TAG: *bytes = Bm * d.W * 4; break;
    case HF_T_POS: *bytes = Bm * 8; break;
    case HF_T_OFFSETS: *bytes = (Bm + 1) * 4; break;
    case HF_T_DRAFT_PROJ: *bytes = Bm * d.S * d.Nd * 4; break;
    case HF_T_DRAFT_MIX: *bytes = Bm * d.S * d.Nz * h->esz; break;
    case HF_T_MEM_X: *bytes = L * Bm * d.Mr * d.dinner * 4; break;
    case HF_T_MEM_B: *bytes = L * Bm * d.Mr * d.N * 4; break;
    case HF_T_MEM_DT: *bytes = L * Bm * d.Hm * d.Mr * 4; break;
    case HF_T_CONV: *bytes = d.blk ? L * Bm * 3 * (d.dinner + d.N) * 4 : 0; break;
    case HF_T_LOGITS: *bytes = d.blk ? Bm * d.S * d.V * 4 : 0; break;
    default: return HF_EINVAL;
  }
  return HF_OK;
}

static const void* tensor_ptr(const hf_handle* h, int which) {
  switch (which) {
    case HF_T_STATE: return h->state;
    case HF_T_RING_K: return h->ring_k;
    case HF_T_RING_V: return h->ring_v;
    case HF_T_RING_TAG: return h->tags;
    case HF_T_POS: return h->pos;
    case HF_T_OFFSETS: return h->offsets;
    case HF_T_DRAFT_PROJ: return h->proj;
    case HF_T_DRAFT_MIX: return h->mix;
    case HF_T_MEM_X: return h->mem_x;
    case HF_T_MEM_B: return h->mem_b;
    case HF_T_MEM_DT: return h->mem_dt;
    case HF_T_CONV: return h->conv_state;
    case HF_T_LOGITS: return h->logits;
  }
  return nullptr;
}

hf_status hf_read_tensor(hf_handle* h, int32_t which, void* host_out, size_t bytes) {
  if (!h) return HF_EINVAL;
  size_t want = 0;
  if (hf_tensor_bytes(h, which, &want) != HF_OK) return fail(h, HF_EINVAL, "unknown tensor id");
  if (!host_out || bytes != want) return fail(h, HF_EINVAL, "host buffer size mismatch");
  HF_CUDA(h, cudaSetDevice(h->device));
  HF_CUDA(h, cudaDeviceSynchronize());
  if (bytes) HF_CUDA(h, cudaMemcpy(host_out, tensor_ptr(h, which), bytes, cudaMemcpyDeviceToHost));
  return HF_OK;
}

// The context: everything a request's drafting depends on (the memory-input
// rows are empty without a memory horizon M > 1, the carried convolution rows
// outside the full block).
static const int kContextTensors[] = {HF_T_STATE, HF_T_RING_K, HF_T_RING_V, HF_T_RING_TAG,
                                      HF_T_POS,   HF_T_MEM_X,  HF_T_MEM_B,  HF_T_MEM_DT,
                                      HF_T_CONV};

size_t hf_context_bytes(const hf_handle* h) {
  if (!h) return 0;
  size_t total = 0, b = 0;
  for (int w : kContextTensors) {
    hf_tensor_bytes(h, w, &b);
    total += b;
  }
  return total;
}

static hf_status copy_context(hf_handle* h, void* host, size_t bytes, bool out) {
  if (!h) return HF_EINVAL;
  if (!host || bytes != hf_context_bytes(h)) return fail(h, HF_EINVAL, "context size mismatch");
  HF_CUDA(h, cudaSetDevice(h->device));
  HF_CUDA(h, cudaDeviceSynchronize());
  size_t off = 0, b = 0;
  for (int w : kContextTensors) {
    hf_tensor_bytes(h, w, &b);
    if (b == 0) continue;
    void* dev = const_cast<void*>(tensor_ptr(h, w));
    if (out)
      HF_CUDA(h, cudaMemcpy(bptr(host, off), dev, b, cudaMemcpyDeviceToHost));
    else
      HF_CUDA(h, cudaMemcpy(dev, bptr(host, off), b, cudaMemcpyHostToDevice));
    off += b;
  }
  return HF_OK;
}

hf_status hf_export_context(hf_handle* h, void* host_out, size_t bytes) {
  return copy_context(h, host_out, bytes, true);
}

hf_status hf_import_context(hf_handle* h, const void* host_in, size_t bytes) {
  return copy_context(h, const_cast<void*>(host_in), bytes, false);
}

hf_status hf_profile_enable(hf_handle* h, int32_t mode) {
  if (!h) return HF_EINVAL;
  if (mode < 0 || mode > 2) return fail(h, HF_EINVAL, "profile mode must be 0, 1 or 2");
  HF_CUDA(h, ensure_device(h));
  if (!h->kept.empty()) {
    HF_CUDA(h, cudaDeviceSynchronize());
    for (auto& r : h->kept) {
      h->pool.push_back(r.a);
      h->pool.push_back(r.b);
    }
    h->kept.clear();
  }
  h->prof = mode;
  // Pre-create events so that recording under stream capture needs no
  // event creation.
  while (mode && h->pool.size() < 256) {
    cudaEvent_t e;
    HF_CUDA(h, cudaEventCreate(&e));
    h->pool.push_back(e);
  }
  return HF_OK;
}

hf_status hf_profile_collect(hf_handle* h) {
  if (!h) return HF_EINVAL;
  HF_CUDA(h, ensure_device(h));
  return collect_profile(h);
}

hf_status hf_profile_read(hf_handle* h, int32_t family, double* total_ms, int64_t* launches,
                          int32_t reset) {
  if (!h || family < 0 || family >= HF_K_COUNT) return HF_EINVAL;
  if (total_ms) *total_ms = h->tot_ms[family];
  if (launches) *launches = h->nl[family];
  if (reset) {
    h->tot_ms[family] = 0;
    h->nl[family] = 0;
  }
  return HF_OK;
}

int64_t hf_launch_count(const hf_handle* h) { return h ? h->launches : 0; }

hf_status hf_debug_set_wait_limit(hf_handle* h, int64_t cycles) {
  const long long lim = cycles < 0 ? hf::kWaitCycles : (long long)cycles;
  if (!h) {
    hf::set_noalloc_wait_limit(lim);
    return HF_OK;
  }
  h->d.wait = lim;
  return HF_OK;
}

hf_status hf_debug_fail_alloc(int64_t k) {
  if (k < 0) return fail(nullptr, HF_EINVAL, "k must be >= 0");
  g_fail_alloc_in.store(k);
  return HF_OK;
}

hf_status hf_debug_check_guards(hf_handle* h) {
  if (!h) return HF_EINVAL;
  HF_CUDA(h, cudaSetDevice(h->device));
  HF_CUDA(h, cudaDeviceSynchronize());
  std::vector<unsigned char> g(kGuardBytes);
  for (size_t i = 0; i < h->allocs.size(); ++i) {
    const char* base = static_cast<const char*>(h->allocs[i]);
    for (int side = 0; side < 2; ++side) {
      const char* at = side == 0 ? base : base + kGuardBytes + h->alloc_bytes[i];
      HF_CUDA(h, cudaMemcpy(g.data(), at, kGuardBytes, cudaMemcpyDeviceToHost));
      for (unsigned char c : g)
        if (c != kGuardByte)
          return fail(h, HF_EDEVICE,
                      "guard region " + std::string(side ? "after" : "before") + " buffer " +
                          std::to_string(i) + " (" + std::to_string(h->alloc_bytes[i]) +
                          " bytes) was overwritten");
    }
  }
  return HF_OK;
}

}  // extern "C"
