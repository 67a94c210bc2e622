/*
 * hyflash.h -- C ABI of the HyFlash drafter-layer library (GB300, sm_103a).
 *
 * What the library computes ("HyFlash: A Prefix-Memory Prior for On-Device
 * Speculative Decoding", abstract; learnaivisually explainer "HyFlash lifts
 * on-device speculative decoding 16.2%", paragraph "That is HyFlash" and FAQ
 * "Why does the memory update only from committed features?"):
 *
 *   Each drafter layer has two branches. Local attention lets the 7 draft-slot
 *   queries attend, in both directions, over a sliding window of the most
 *   recent committed target features and over all draft slots. A Mamba-2
 *   recurrent memory folds committed target features into a fixed-size state
 *     h_t = exp(dt_t * A) * h_{t-1} + dt_t * x_t (outer) B_t,   y = C . h
 *   (dt = softplus(f W_dt + dt_bias), A = -exp(A_log)); drafting only reads
 *   it, and only features the target committed ever write it.
 *
 *   prefill : fold a committed prefix into the memory, fill the window.
 *   commit  : append the accepted features of one verification round to the
 *             window ring and advance the memory over them, in order.
 *   draft   : run the layers for the 7 slot embeddings; read-only.
 *
 * Readings where the pages are silent (the oracle states the same ones):
 * out = X + O W_o + y W_mo (two branches summed into the residual, no norms,
 * RoPE, MLP, conv1d, gate or skip); the draft-time memory query is
 * C_s = X_s W_C; window K/V and memory inputs are projections of the
 * committed target features by the layer's own weights; one SSM group;
 * softmax scale 1/sqrt(head_dim); a slot attends to its own key too; GQA
 * maps query head h to KV head h / (n_q_heads / n_kv_heads); committed
 * position t lives in ring slot t mod window.
 *
 * Conventions for every call below:
 *   - "device" pointers are CUDA global-memory addresses on the handle's
 *     device, "host" pointers are ordinary CPU memory. The caller owns every
 *     buffer it passes; the library owns the window rings, recurrent states,
 *     positions, weights and its scratch.
 *   - Matrices are row-major. Element type of features, slot embeddings,
 *     outputs and weights is the handle's dtype (fp32 or bf16);
 *     dt_bias and A_log are always fp32; the recurrent state is always fp32.
 *     Device buffers passed to prefill, commit and draft must be 16-byte
 *     aligned (HF_EINVAL otherwise); d_model must be a multiple of 8.
 *   - Kernels are launched with programmatic dependent launch: each kernel
 *     of a call may start while the previous one finishes, and waits for
 *     it before touching its data. Calls may be captured into CUDA graphs
 *     (nothing in prefill/commit/draft allocates or synchronises).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued asynchronously; nothing here synchronises the
 *     host unless its comment says so.
 *   - Errors found on the host return at once and change nothing. Errors
 *     found on the device (an accepted count outside 0..block+1) leave that
 *     request untouched, set the handle's device error word, and surface at
 *     the next hf_sync(). hf_last_error() gives a message for the last
 *     non-OK status.
 *   - A handle is not thread-safe; calls on one handle must be ordered.
 */
#ifndef HYFLASH_H
#define HYFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hf_handle hf_handle;

typedef enum {
  HF_OK = 0,
  HF_EINVAL = 1,   /* bad argument or configuration */
  HF_ENOMEM = 2,   /* device allocation failed (nothing leaked) */
  HF_ECUDA = 3,    /* CUDA runtime error (no device, launch failure, ...) */
  HF_ETIMEOUT = 4, /* a bounded device-side wait gave up */
  HF_EDEVICE = 5   /* a device-side argument check failed (see hf_last_error) */
} hf_status;

typedef enum { HF_F32 = 0, HF_BF16 = 1 } hf_dtype;

/* Shape of the drafter. Block is the number of draft slots (7 on the pages:
 * "In the paper the block is 7 positions"); commits take up to block+1 rows
 * (7 drafts plus the target's bonus token). */
typedef struct {
  int32_t d_model;      /* D */
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* Hkv, divides Hq */
  int32_t head_dim;     /* dh: 32, 64, 128 or 256 */
  int32_t window;       /* W >= block+1: sliding-window ring length */
  int32_t block;        /* S = 7 draft slots (1..16 accepted) */
  int32_t ssm_heads;    /* Hm */
  int32_t ssm_headdim;  /* P, multiple of 4; P*N a multiple of 128, <= 8192 */
  int32_t d_state;      /* N, a power of two in 4..128 */
  int32_t n_groups;     /* must be 1 */
  int32_t n_layers;     /* drafter depth */
  int32_t max_batch;    /* requests held by the handle */
  int32_t chunk;        /* prefill scan chunk length: 64, 128 or 256 */
  int32_t dtype;        /* hf_dtype */
  int64_t prefill_tokens_max; /* tokens per internal prefill pass; 0 = 16384 */
  /* Ablation modes of the paper's intervention table (HyFlash paper, table
   * "Recurrent history" / "Intra-block interactions"), 0 = off:
   *   cross_slot_off = 1: attention among the draft slots is switched off --
   *     slot s attends to the window entries and to its own key only
   *     ("Cross-slot off");
   *   mem_horizon = M > 0: the memory holds the fold, from zero, of the last
   *     M committed features only ("SSM: Last 512" is M = 512, "SSM: Last
   *     feature" M = 1); M <= window. For M > 1 the handle keeps the x, B
   *     and dt rows of the last M + block + 1 committed features per request
   *     and layer, and each commit removes the contribution of the features
   *     that leave the horizon. */
  int32_t cross_slot_off;
  int32_t mem_horizon;
  /* Memory kind: HF_MEM_MAMBA2 (the pages' Mamba-2 memory) or
   * HF_MEM_GATED_DELTA (the paper's swap to Gated DeltaNet-2, memory-swap
   * table): per head S <- S (alpha (I - beta k k^T)) + beta v k^T with unit
   * keys k = B/|B|, values x, alpha = exp(dt A) as in Mamba-2, beta =
   * sigmoid(f W_beta), and the draft-time read y = S C/|C| (the gated delta
   * rule of "Gated Delta Networks: Improving Mamba2 with Delta Rule").
   * Needs w_beta; no memory horizon. */
  int32_t memory_kind;
  /* Weight precision: 16 (the model dtype) or 4 (bf16 handles only; the
   * paper's INT4 / GPTQ drafter): weights enter through hf_set_weights_q4 as
   * 4-bit codes with a bf16 scale and an integer zero point per output
   * column and group of 128 input rows, w = scale * (code - zero). Draft and
   * commit products of at most 32 activation rows read the 4-bit tiles and
   * dequantise them on chip; wider products and prefill use the same
   * weights dequantised once to bf16. d_model, n_q_heads*head_dim and
   * ssm_heads*ssm_headdim must be multiples of 128. 0 means 16. */
  int32_t weight_bits;
  /* Full drafter block around the layer (0: the layer alone, as above; 1:
   * the block). The pages describe each drafter layer's two branches and
   * name none of the parts around them; the block takes the plainest
   * reading of the model families they use (Qwen3 targets, Mamba-2):
   *   a = RMSNorm(X; g_mix)                       (eps 1e-6, one norm for both branches)
   *   Q, K_s at positions pos + s by rotate-half RoPE (base 1e6); committed
   *     keys are rotated at their positions when they enter the ring
   *   the memory's x and B pass Mamba-2's causal depthwise conv1d (width 4,
   *     bias, SiLU) with the last 3 pre-conv committed rows carried across
   *     commits; dt is not convolved; the draft-time C is not either
   *   y_s = (C_s h + D[head] x_s) * silu(z_s), x_s = a W_x, z_s = a W_z
   *   X1 = X + O W_o + y W_mo;  out = X1 + W_down(silu(n W_gate) * (n W_up)),
   *     n = RMSNorm(X1; g_mlp)
   *   hf_draft_tokens: logits = RMSNorm(out; g_final) W_lm and the argmax
   *     token of every slot (ties to the lowest id).
   * Weights through hf_set_block_weights and hf_set_head_weights. Needs the
   * Mamba-2 memory, no memory horizon, weight_bits 16, mlp_dim a multiple
   * of 8, vocab >= 2. */
  int32_t block_kind;
  int32_t mlp_dim;      /* F: SwiGLU width (block only) */
  int32_t vocab;        /* V: LM-head rows (block only) */
} hf_config;

enum { HF_LAYER = 0, HF_FULL_BLOCK = 1 };

enum { HF_MEM_MAMBA2 = 0, HF_MEM_GATED_DELTA = 1 };

/* One layer's weights, HOST pointers, row-major [in, out] in the handle's
 * dtype (dt_bias, A_log: fp32 [ssm_heads]). Shapes:
 *   w_q [D, Hq*dh]  w_k, w_v [D, Hkv*dh]  w_o [Hq*dh, D]
 *   w_x [D, Hm*P]   w_B, w_C [D, N]       w_dt [D, Hm]   w_mo [Hm*P, D]
 *   w_beta [D, Hm] (gated-delta memory only) */
typedef struct {
  const void* w_q;
  const void* w_k;
  const void* w_v;
  const void* w_o;
  const void* w_x;
  const void* w_B;
  const void* w_C;
  const void* w_dt;
  const void* w_mo;
  const float* dt_bias;
  const float* A_log;
  const void* w_beta;  /* [D, Hm]: gated-delta writing strength (NULL otherwise) */
} hf_layer_weights;

/* The block's parts around one layer (block_kind = HF_FULL_BLOCK), HOST
 * pointers, row-major [in, out]: gains g_mix, g_mlp fp32 [D]; w_z [D, Hm*P]
 * (model dtype); d_skip fp32 [Hm]; conv_w fp32 [Hm*P + N, 4] (tap 3 on the
 * newest row) and conv_b fp32 [Hm*P + N] over the x | B channels; w_gate,
 * w_up [D, F], w_down [F, D] (model dtype). */
typedef struct {
  const float* g_mix;
  const float* g_mlp;
  const void* w_z;
  const float* d_skip;
  const float* conv_w;
  const float* conv_b;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
} hf_block_weights;

/* One 4-bit matrix of hf_layer_weights_q4, HOST pointers, for a weight of
 * shape [in, out] (in a multiple of 128): codes uint8 [in, out] with values
 * 0..15; scales bf16 bits [in/128, out]; zeros uint8 [in/128, out] (0..15).
 * Element (i, o) is scales[i/128][o] * (codes[i][o] - zeros[i/128][o]). */
typedef struct {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint8_t* zeros;
} hf_q4_matrix;

/* A layer's weights in 4 bits (same matrices and shapes as
 * hf_layer_weights; w_beta only with the gated-delta memory, else codes
 * NULL). dt_bias and A_log stay fp32 [ssm_heads]. */
typedef struct {
  hf_q4_matrix w_q, w_k, w_v, w_o, w_x, w_B, w_C, w_dt, w_mo, w_beta;
  const float* dt_bias;
  const float* A_log;
} hf_layer_weights_q4;

/* Create a handle on CUDA device `device`: validates cfg (HF_EINVAL before
 * touching CUDA), allocates and zeroes rings, states, positions, weights and
 * scratch (HF_ENOMEM on failure, everything freed). Synchronises. */
hf_status hf_create(const hf_config* cfg, int32_t device, hf_handle** out);

/* Free everything the handle owns. Synchronises the device. NULL is a no-op. */
void hf_destroy(hf_handle* h);

/* Copy one layer's weights in from HOST memory (re-laid-out for the kernels:
 * transposed to [out, in] and concatenated per call site). Synchronises;
 * the caller may free its buffers afterwards. */
hf_status hf_set_weights(hf_handle* h, int32_t layer, const hf_layer_weights* w);

/* The same for a handle with weight_bits = 4 (HF_EINVAL otherwise, and for
 * codes or zeros above 15): keeps the 4-bit tiles of the skinny products and
 * the bf16 dequantisation of the others. Synchronises. */
hf_status hf_set_weights_q4(hf_handle* h, int32_t layer, const hf_layer_weights_q4* w);

/* A block handle's weights of one layer: the layer's (as hf_set_weights)
 * and the block's parts around it. HOST pointers; synchronises. HF_EINVAL on
 * a handle without the block (and hf_set_weights is refused on one with it). */
hf_status hf_set_block_weights(hf_handle* h, int32_t layer, const hf_layer_weights* w,
                               const hf_block_weights* bw);

/* The LM head of a block handle: g_final fp32 [D], w_lm [D, vocab] in the
 * model dtype, HOST pointers. Synchronises. */
hf_status hf_set_head_weights(hf_handle* h, const float* g_final, const void* w_lm);

/* Prefill (fold the committed prefix). feats: DEVICE [sum(lens), D] packed
 * in request order; lens: HOST int32 [n_req], each >= 0; requests: HOST int32
 * [n_req] distinct request slots in 0..max_batch-1, or NULL for 0..n_req-1.
 * Each named request is reset, its memory becomes the fold of all its
 * features from h = 0 (chunked scan, chunk = cfg.chunk), its window holds the
 * last min(L, W) features' K/V at slot pos mod W, and pos = L. Other
 * requests are untouched. */
hf_status hf_prefill(hf_handle* h, const void* feats, const int32_t* lens,
                     const int32_t* requests, int32_t n_req, void* stream);

/* Commit one verification round for requests 0..batch-1. feats: DEVICE
 * [batch, block+1, D]; n_accepted: DEVICE int32 [batch]. For request b the
 * rows t < n_b are appended in order (ring slot (pos_b + t) mod W, memory
 * update token by token) and pos_b += n_b. Rows t >= n_b (the rejected
 * drafts) pass through the batched projection but are discarded: they never
 * reach the window, the memory or the positions. n_b = 0 is a no-op. n_b outside 0..block+1 leaves request b untouched and
 * raises HF_EDEVICE at the next hf_sync. Packed row offsets (exclusive scan
 * of the valid counts) are kept for inspection (HF_T_OFFSETS). */
hf_status hf_commit(hf_handle* h, const void* feats, const int32_t* n_accepted,
                    int32_t batch, void* stream);

/* Draft for requests 0..batch-1: slot_emb DEVICE [batch, block, D] ->
 * out DEVICE [batch, block, D] (may not alias slot_emb). Runs every layer;
 * layer l+1's slot input is layer l's output. Never writes rings, states or
 * positions. */
hf_status hf_draft(hf_handle* h, const void* slot_emb, void* out, int32_t batch,
                   void* stream);

/* hf_draft followed by the LM head (block handles with head weights):
 * out DEVICE [batch, block, D] as hf_draft, and tokens DEVICE int32
 * [batch, block]: the argmax of each slot's logits (ties to the lowest
 * token id); the logits stay readable as HF_T_LOGITS. */
hf_status hf_draft_tokens(hf_handle* h, const void* slot_emb, void* out, int32_t* tokens,
                          int32_t batch, void* stream);

/* One serving iteration: commit the verified round (feats, n_accepted as in
 * hf_commit), then draft the next block (slot_emb, out as in hf_draft). The
 * result -- context and out -- is exactly that of hf_commit followed by
 * hf_draft (the HyFlash explainer, "That is HyFlash": the memory and the
 * window take the newly committed features, then the parallel block is
 * drafted against them). bf16 handles run it as one pipeline: the commit
 * projection and the first layer's slot projection stream their weights in
 * one grouped launch (at a batch whose commit product alone has a 128 x 256
 * tile per SM: the commit projection on the persistent GEMM, then the slot
 * projection, whose main loop runs beside the commit projection's last
 * tiles), and at large batch the first layer's memory read is computed on
 * the updated state inside the state update (the state is read once per
 * round). Other handles call the two entry points in turn. */
hf_status hf_round(hf_handle* h, const void* feats, const int32_t* n_accepted,
                   const void* slot_emb, void* out, int32_t batch, void* stream);

/* Synchronise `stream`, then read and clear the device error word. Returns
 * HF_EDEVICE if a device-side check failed since the last hf_sync, HF_ECUDA
 * on an asynchronous CUDA error, HF_OK otherwise. */
hf_status hf_sync(hf_handle* h, void* stream);

/* Message for the last non-OK status of this handle ("" if none); the
 * pointer stays valid until the next call on the handle. h may be NULL
 * (then the message of the last failed call without a handle -- hf_create
 * or hf_attention_noalloc -- in this thread). */
const char* hf_last_error(const hf_handle* h);

/* Static name of a status code. */
const char* hf_status_string(hf_status s);

/* ---- inspection (tests, checkpoints) ---------------------------------- */

typedef enum {
  HF_T_STATE = 0,     /* fp32 [L, max_batch, Hm, P, N] */
  HF_T_RING_K = 1,    /* dtype [L, max_batch, Hkv, W, dh] */
  HF_T_RING_V = 2,    /* dtype [L, max_batch, Hkv, W, dh] */
  HF_T_RING_TAG = 3,  /* int32 [max_batch, W]: committed position held by
                         each slot, -1 if empty */
  HF_T_POS = 4,       /* int64 [max_batch]: committed tokens per request */
  HF_T_OFFSETS = 5,   /* int32 [max_batch + 1]: packed row offsets of the
                         last commit (entries past its batch are stale) */
  HF_T_DRAFT_PROJ = 6,/* fp32 [max_batch*block, Hq*dh + 2*Hkv*dh + N]: last
                         layer's slot projections Q|K_s|V_s|C_s, last draft
                         (full block: + x_s | z_s, Hm*P each; Q and K_s
                         rotated) */
  HF_T_DRAFT_MIX = 7, /* dtype [max_batch*block, Hq*dh + Hm*P]: last layer's
                         attention output | memory read y, last draft (full
                         block: y after the skip and the gate) */
  /* memory horizon M > 1 only (0 bytes otherwise); R = M + block + 1 ring
   * rows, committed position t in row t mod R */
  HF_T_MEM_X = 8,     /* fp32 [L, max_batch, R, Hm*P]: x of the last features */
  HF_T_MEM_B = 9,     /* fp32 [L, max_batch, R, N]: B of the last features */
  HF_T_MEM_DT = 10,   /* fp32 [L, max_batch, Hm, R]: dt (after softplus) */
  /* full block only (0 bytes otherwise) */
  HF_T_CONV = 11,     /* fp32 [L, max_batch, 3, Hm*P + N]: last 3 pre-conv
                         committed x | B rows, oldest first */
  HF_T_LOGITS = 12    /* fp32 [max_batch*block, vocab]: last hf_draft_tokens */
} hf_tensor_id;

/* Size in bytes of an inspectable tensor. */
hf_status hf_tensor_bytes(const hf_handle* h, int32_t which, size_t* bytes);

/* Copy a whole inspectable tensor to HOST memory (bytes must equal
 * hf_tensor_bytes). Synchronises the device. */
hf_status hf_read_tensor(hf_handle* h, int32_t which, void* host_out, size_t bytes);

/* Bytes of the complete drafter context (states, rings, tags, positions,
 * with a memory horizon M > 1 the x/B/dt rows of the last features, and in
 * a full block the convolution's carried rows):
 * the fixed-size draft-side memory of all requests and layers. */
size_t hf_context_bytes(const hf_handle* h);

/* Copy the complete context to / from HOST memory (checkpoint, or byte
 * comparison of before/after). Synchronise the device. */
hf_status hf_export_context(hf_handle* h, void* host_out, size_t bytes);
hf_status hf_import_context(hf_handle* h, const void* host_in, size_t bytes);

/* ---- measurement ------------------------------------------------------ */

/* Kernel families timed by the profiler and counted by hf_launch_count. */
typedef enum {
  HF_K_DRAFT_PROJ = 0,   /* draft input projections (Q|K_s|V_s|C_s) */
  HF_K_ATTN_MEM = 1,     /* window+block attention and memory read */
  HF_K_OUT_PROJ = 2,     /* output projections + residual */
  HF_K_ROUND_PROJ = 3,   /* hf_round: commit + first slot projection (one or two launches) */
  HF_K_COMMIT_PROJ = 4,  /* commit projections + ring append */
  HF_K_COMMIT_STATE = 5, /* sequential memory update */
  HF_K_PREFILL = 6,      /* every prefill kernel */
  HF_K_OTHER = 7,        /* split-K combine and helpers; full block: norms,
                            RoPE, gate/skip */
  HF_K_MLP = 8,          /* full block: SwiGLU MLP */
  HF_K_HEAD = 9,         /* full block: LM head and argmax */
  HF_K_COUNT = 10
} hf_kernel_family;

/* Per-kernel-family timing with CUDA events recorded on the launch stream
 * around each family's launches. mode 0: off. mode 1: every call records
 * fresh events, read once by hf_profile_collect. mode 2 (for CUDA graphs):
 * events are recorded as external event nodes (cudaEventRecordExternal), so
 * calls captured into a graph re-record them on every replay; the records
 * are kept, and each hf_profile_collect adds the latest replay's times.
 * Changing the mode synchronises the device and drops kept records: do it
 * only when no graph holding them will be replayed again. */
hf_status hf_profile_enable(hf_handle* h, int32_t mode);

/* Synchronise on the recorded events and add their elapsed times and
 * launch counts to the per-family totals. */
hf_status hf_profile_collect(hf_handle* h);

/* Per-family totals (milliseconds, launches) accumulated by
 * hf_profile_collect; reset != 0 zeroes that family afterwards. */
hf_status hf_profile_read(hf_handle* h, int32_t family, double* total_ms,
                          int64_t* launches, int32_t reset);

/* Number of kernels this handle has launched since creation. */
int64_t hf_launch_count(const hf_handle* h);

/* ---- failure detection (tests) ---------------------------------------
 *
 * Hooks that let tests drive the error paths without faulting a GPU. */

/* Limit, in clock cycles, of the ring-tile wait of the CUDA-core attention
 * kernel (the fp32 path of hf_draft / hf_round) of handle h; with h NULL,
 * of hf_attention_noalloc's ring-tile wait. cycles < 0 restores the default
 * (about 2 s); 0 makes that wait give up at once, so the kernel takes its
 * expiry path: it raises the timeout bit, lets its copies land (default
 * limit), drops its ring tile (the window is left out of that draft) and
 * returns; hf_sync then reports HF_ETIMEOUT and clears the word. Never
 * fails. */
hf_status hf_debug_set_wait_limit(hf_handle* h, int64_t cycles);

/* Make the k-th device allocation made by the library from now on fail as
 * if the device were out of memory (k >= 1; 0 switches it off). hf_create
 * then returns HF_ENOMEM and frees whatever it had allocated. Process-wide. */
hf_status hf_debug_fail_alloc(int64_t k);

/* Every device buffer of a handle sits between two 256-byte guard regions
 * filled with 0xA5. Synchronises the device and reads them all back:
 * HF_OK if intact, HF_EDEVICE naming the first overwritten one. */
hf_status hf_debug_check_guards(hf_handle* h);

/* ---- allocation-free window attention --------------------------------
 *
 * The pages have no counterpart to this call. It computes the window+block
 * attention of hf_draft (every slot query of a request over the valid ring
 * entries and the block's slot keys) with a separate split-combine kernel:
 * the window is cut into 32-key splits, one CTA each, whose partial results
 * go to one fixed array compiled into the library's device image (not to
 * memory a handle allocated), and the last split of each (request, KV head)
 * to finish combines them in split order. hf_draft itself runs a cluster
 * kernel that combines on chip; the two agree to rounding.
 *
 * It is for callers that cannot allocate device memory when they run the
 * op: a host that hands all of the GPU's memory to its own arena, a serving
 * loop whose memory was sized once at start-up, or code that must not
 * cause the device-wide synchronisation cudaMalloc/cudaFree can bring. This
 * call makes no cudaMalloc, cudaFree or other allocating call.
 *
 * The fixed array holds 4,194,304 floats (16 MiB) and exists on every GPU
 * that loads the library until the process exits. A call needs
 *   batch * n_kv_heads * ceil(window / 32) * (n_q_heads / n_kv_heads)
 *         * block * (head_dim + 2)
 * floats of it, and batch * n_kv_heads <= 16384; a larger call returns
 * HF_EINVAL and launches nothing. So does a call whose CTA would need more
 * shared memory than the device allows per block: about
 *   (n_q_heads/n_kv_heads) * block * (4 (head_dim + 4) + 4 (32 + block)
 *     + 4 ceil(window/32)) + 8 (32 + block)(head_dim + 4) + 64 head_dim e
 * bytes (e = 4 for HF_F32, 2 for HF_BF16) against 232,448 on GB300.
 * All calls share the one array: calls that can overlap on the GPU (other
 * streams, other host threads) race and must be ordered by the caller. Each
 * call rewrites every partial it later reads, so nothing needs clearing.
 * The first call on each device looks up the array's device address and the
 * device's shared-memory limit (once, with that device current); make that
 * first call before any stream capture.
 *
 * Arguments (all buffers DEVICE memory on the current device, caller-owned):
 *   dtype     HF_F32 or HF_BF16: element type of ring_k, ring_v and out.
 *   proj      fp32 [batch*block, proj_ld]: row b*block+s holds slot s of
 *             request b: query head h at columns [h*dh, (h+1)*dh), slot key
 *             of KV head g at Hq*dh + g*dh, slot value at Hq*dh + Hkv*dh + g*dh
 *             (proj_ld >= Hq*dh + 2*Hkv*dh; the draft projection layout).
 *   ring_k/v  [batch, Hkv, window, dh]: window entries; the first
 *             min(pos_b, window) slots of request b are attended.
 *   pos       int64 [batch]: committed tokens per request.
 *   out       [batch*block, out_ld]: attention output of head h written to
 *             columns [h*dh, (h+1)*dh) (out_ld >= Hq*dh); other columns kept.
 *   status    int32, optional (NULL: not reported): if a ring-tile copy does
 *             not land within the wait limit (about 2 s), the CTA records
 *             HF_ETIMEOUT's device bit (2) here with an atomic OR, waits once
 *             more (bounded) for its copies, and leaves its split out of the
 *             result. The caller zeroes it and reads it when it likes.
 * Errors: HF_EINVAL for bad sizes or pointers (message in
 * hf_last_error(NULL)), HF_ECUDA for a failed launch. */
hf_status hf_attention_noalloc(int32_t dtype, int32_t batch, int32_t n_q_heads,
                               int32_t n_kv_heads, int32_t head_dim, int32_t window,
                               int32_t block, const float* proj, int32_t proj_ld,
                               const void* ring_k, const void* ring_v, const int64_t* pos,
                               void* out, int32_t out_ld, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HYFLASH_H */
