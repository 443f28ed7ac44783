/*
 * dflash.h - C ABI of the DFlash drafter pass on one NVIDIA GB300 (sm_103a).
 *
 * The library implements the data-parallel hot path of DFlash block-diffusion
 * speculative decoding ("DFlash - Block Diffusion for Flash Speculative
 * Decoding", notes on the paper, sections 4.2-4.5):
 *
 *   dflash_fuse_ctx  fuses the target model's multi-layer hidden features
 *                    (section 4.2, fusion equation) and injects them as K/V
 *                    into every drafter layer's context cache (section 4.3,
 *                    the K_i / V_i equations);
 *   dflash_draft     runs one non-causal pass over [anchor, MASK x (B-1)] and
 *                    returns B-1 greedy draft ids (section 4.4);
 *   dflash_verify    greedy acceptance against the target's argmax ids with
 *                    the bonus token, then commit / roll back the cache
 *                    (section 4.5; tau as defined in section 2.2).
 *
 * Conventions (all entry points):
 *  - Every call returns a dflash_status. Nothing throws across the ABI.
 *    dflash_last_error() describes the last failure of a context.
 *  - Tensors named "device" are caller-owned device pointers; tensors named
 *    "host" are caller-owned host pointers. The library never frees either.
 *  - Floating-point tensors are bf16 (passed as uint16_t bit patterns) or
 *    fp32 where stated; ids are int32.
 *  - Matrices are row-major, weights in nn.Linear layout [out, in].
 *  - Calls that take a cudaStream_t (passed as void*) are asynchronous on that
 *    stream and never synchronise the host. One context must be driven from
 *    one stream at a time. Device-side faults that kernels detect (a bounded
 *    wait that ran out, an index out of range) are latched in a status word
 *    that dflash_sync() reports.
 *  - Weights are borrowed: they must stay valid and unchanged for the life of
 *    the context. The library owns the KV pool, page tables and workspaces it
 *    allocates in dflash_create().
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFLASH_OK = 0,
  DFLASH_EINVAL = 1,   /* bad argument; nothing was enqueued                  */
  DFLASH_ENOMEM = 2,   /* KV page pool or device memory exhausted              */
  DFLASH_ECUDA = 3,    /* a CUDA runtime call failed                           */
  DFLASH_ETIMEOUT = 4, /* a kernel's bounded wait ran out (reported by sync)   */
  DFLASH_EDEVICE = 5   /* a kernel detected an out-of-range index (by sync)    */
} dflash_status;

typedef struct dflash_ctx dflash_ctx;

/* Drafter shape and capacity. Shape fields follow the DFlash notes' setup
 * (5 drafter layers, 5 fused target layers, block size 16) but any values
 * meeting the stated constraints are accepted. */
typedef struct {
  int hidden;          /* H; multiple of 64                                          */
  int n_heads;         /* query heads; n_heads * head_dim multiple of 128            */
  int n_kv_heads;      /* kv heads; divides n_heads; n_kv_heads * head_dim mult. 128  */
  int head_dim;        /* d: 64 or 128                                               */
  int ffn;             /* F: SwiGLU width; multiple of 8                             */
  int vocab;           /* V: shared embedding / LM head rows                         */
  int n_layers;        /* L drafter layers, 1..16                                    */
  int n_feat_layers;   /* L_f target layers fused by W_c, 1..16                       */
  float rope_base;     /* RoPE theta base (rotate-half pairing (i, i+d/2))            */
  float rms_eps;       /* RMSNorm epsilon                                            */
  int mask_id;         /* id of the MASK token                                       */
  int max_seqs;        /* sequence slots: seq ids are 0..max_seqs-1                   */
  int max_batch;       /* most sequences in one call, 1..64                          */
  int max_block;       /* largest block B, 1..32                                     */
  int max_ctx;         /* most cached tokens per sequence (committed + pending)      */
  int max_pages;       /* KV pool size in 64-token pages (shared by all sequences)   */
  int max_fuse_tokens; /* most feature rows in one dflash_fuse_ctx call               */
  int kv_format;       /* cached context K/V: 0 bf16; 1 8-bit blocks (q8_0: per head
                          row, blocks of 32 values, int8 codes round(x/d) halves away
                          from zero, d = max|x|/127 stored as fp16); drafter only  */
} dflash_config;

/* One drafter layer's weights, device pointers to bf16 (nn.Linear layout). */
typedef struct {
  const uint16_t* w_q;    /* [n_heads*d,    H]                      */
  const uint16_t* w_k;    /* [n_kv_heads*d, H]  also projects H_t   */
  const uint16_t* w_v;    /* [n_kv_heads*d, H]  also projects H_t   */
  const uint16_t* w_o;    /* [H, n_heads*d]                         */
  const uint16_t* w_gate; /* [F, H]                                 */
  const uint16_t* w_up;   /* [F, H]                                 */
  const uint16_t* w_down; /* [H, F]                                 */
  const uint16_t* g_attn; /* [H] input RMSNorm gain                 */
  const uint16_t* g_ffn;  /* [H] post-attention RMSNorm gain        */
} dflash_layer_weights;

/* All drafter weights, device pointers to bf16. `layers` is a HOST array of
 * n_layers entries (copied by dflash_create). */
typedef struct {
  const uint16_t* w_c;     /* [H, L_f*H] shared fusion projection W_c        */
  const uint16_t* g_c;     /* [H] fusion RMSNorm gain                        */
  const uint16_t* embed;   /* [V, H] shared token embedding                  */
  const uint16_t* lm_head; /* [V, H] shared LM head                          */
  const uint16_t* g_final; /* [H] final RMSNorm gain                         */
  const dflash_layer_weights* layers;
} dflash_weights;

/* Create a context on the current CUDA device: validates the config,
 * allocates the KV pool (n_layers * max_pages * 2 * n_kv_heads * 64 * d bf16,
 * zero-filled), page tables, RoPE table and workspaces, and encodes TMA
 * descriptors for the weights. Synchronises the device.
 * Errors: EINVAL (config out of range, null pointer, weight not 16-byte
 * aligned), ENOMEM, ECUDA. On error *out is NULL. */
dflash_status dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_ctx** out);

/* Synchronise the device and free everything the context allocated. */
dflash_status dflash_destroy(dflash_ctx* ctx);

/* Static description of the last error of ctx (or of the last failed
 * dflash_create when ctx is NULL). Never NULL. */
const char* dflash_last_error(const dflash_ctx* ctx);

/* Forget sequence `seq`: committed and pending lengths become 0 and its pages
 * return to the pool. Synchronises the device. EINVAL if seq is out of range. */
dflash_status dflash_seq_reset(dflash_ctx* ctx, int seq);

/* Exact committed and pending lengths of `seq`. Synchronises the device.
 * Either output pointer may be NULL. */
dflash_status dflash_seq_len(dflash_ctx* ctx, int seq, int* committed, int* pending);

/* Append fused target features to the drafter's context cache (KV injection).
 *
 * DFlash notes 4.2-4.3: H_t = RMSNorm(W_c [H^(l1); ...; H^(lLf)]) per token,
 * then for every layer i: K_i = RoPE(W_i^K H_t), V_i = W_i^V H_t, written to
 * the paged cache at the token's absolute position.
 *
 *  seq_ids  host  [n_seq]       distinct sequence slots
 *  n_new    host  [n_seq]       tokens appended per sequence (>= 0)
 *  feats    device [sum(n_new), L_f*H] bf16, rows grouped by sequence in
 *           seq_ids order; each row is the target's hidden states of L_f
 *           layers, layer-major (shallow to deep).
 *  pending  0: the tokens are committed at once (sequence must have no pending
 *              tokens); 1: the tokens are speculative until the next
 *              dflash_verify, which commits the first tau of them.
 * Positions: the i-th new token of a sequence goes to position
 * committed + pending + i. Errors: EINVAL (n_seq > max_batch, sum(n_new) >
 * max_fuse_tokens, length would exceed max_ctx, duplicate seq, committed
 * append with pending tokens), ENOMEM (page pool exhausted; nothing enqueued).
 */
dflash_status dflash_fuse_ctx(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq,
                              const int32_t* n_new, const uint16_t* feats, int pending,
                              void* stream);

/* One parallel drafting pass (DFlash notes 4.4): for each sequence the block
 * [anchor, MASK x (B-1)] at positions committed .. committed+B-1 runs once
 * through every drafter layer, attending without a causal mask to itself and
 * to the sequence's committed injected context; the final RMSNorm and the
 * shared LM head score every masked position and the greedy (argmax, lowest
 * index on ties) id is returned. Pending tokens are not attended.
 *
 *  seq_ids    host   [n_seq]
 *  anchor_ids device [n_seq] int32, the last verified token of each sequence
 *  B          1..max_block (B = 1 runs the layers and returns no ids)
 *  draft_ids  device [n_seq, B-1] int32 output
 * Errors: EINVAL. */
dflash_status dflash_draft(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq,
                           const int32_t* anchor_ids, int B, int32_t* draft_ids,
                           void* stream);

/* Greedy verify and commit (DFlash notes 4.5): per sequence,
 * a = number of leading j in 0..B-2 with draft[j] == target[j] (draft[j] is
 * the drafter's id for block position j+1, target[j] the target's greedy id
 * after block position j); tau = a + 1, bonus = target[a]. Then the first
 * min(tau, pending) pending tokens are committed and the rest discarded.
 *
 *  draft_ids  device [n_seq, B-1] int32
 *  target_ids device [n_seq, B]   int32
 *  tau, bonus device [n_seq]      int32 outputs
 * Errors: EINVAL. */
dflash_status dflash_verify(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, int B,
                            const int32_t* draft_ids, const int32_t* target_ids,
                            int32_t* tau, int32_t* bonus, void* stream);

/* ---- the target side of the cycle: a target-shaped verify pass ----
 * The DFlash notes' decoding cycle (4.5, "The Decoding Loop"): the target LLM
 * computes logits for all positions of the drafted block in one batched
 * forward pass, its greedy choice after each position feeds the acceptance
 * check, and (4.2, 6.1 "Setup") the hidden states of 5 of its layers,
 * uniformly sampled between layer 2 and the third-to-last, are the drafter's
 * features. The time of that pass is T_verify of the speedup formula (2.2);
 * the same pass over one token is a plain decoding step (L_target).
 *
 * A target context is a dflash_ctx built by dflash_target_create: the
 * drafter's pre-norm layer (RMSNorm, rotate-half RoPE, GQA, SwiGLU; no
 * QK-norm) with causal attention, caching its own K/V in the same paged
 * layout. dflash_verify, dflash_seq_len, dflash_seq_reset, dflash_sync and
 * the inspection hooks work on it as on a drafter; dflash_fuse_ctx,
 * dflash_draft, dflash_draft_sample and dflash_set_path_selector return
 * EINVAL. */

/* The default feature layers: out[k] = (0-based) index of 1-based layer
 * round(2 + k (n_layers - 4) / (n_feat - 1)), k < n_feat (n_feat = 1: layer
 * 2); for 36 layers and 5 features, 1-based layers 2, 10, 18, 26, 34.
 * Host only. Errors: EINVAL (n_layers < 5, n_feat outside 1..min(16,
 * n_layers - 3), out NULL). */
dflash_status dflash_target_feature_layers(int n_layers, int n_feat, int32_t* out);

/* Create a target context. cfg as for dflash_create, except: n_layers up to
 * 64; n_feat_layers = number of feature layers (0..16); mask_id and
 * max_fuse_tokens unused. w as for dflash_create without the fusion weights
 * (w_c, g_c ignored). feat_layers: host [n_feat_layers] strictly increasing
 * 0-based layer indices (may be NULL when n_feat_layers is 0).
 * Errors: as dflash_create. */
dflash_status dflash_target_create(const dflash_config* cfg, const dflash_weights* w, const int32_t* feat_layers,
                                   dflash_ctx** out);

/* One target pass per sequence over block_ids (B tokens at positions
 * committed .. committed+B-1; the sequence must have no pending tokens):
 * causal attention over its cached tokens and the block, the block's K/V
 * appended to its cache (pending = 1: speculative until dflash_verify, which
 * commits the first min(tau, B); pending = 0: committed at once, as in
 * prefill), and the argmax of the logits at every block position.
 *  block_ids  device [n_seq, B] int32
 *  B          1..max_block
 *  target_ids device [n_seq, B] int32 output: t_j, the greedy token after
 *             block position j (dflash_verify's target_ids)
 *  feats      device [n_seq * B, n_feat_layers * H] bf16 output, 16-byte
 *             aligned, or NULL: each block position's residual stream after
 *             each feature layer, layer-major (dflash_fuse_ctx's feats)
 * Errors: EINVAL, ENOMEM (page pool exhausted; nothing enqueued). */
dflash_status dflash_target_forward(dflash_ctx* t, const int32_t* seq_ids, int n_seq, const int32_t* block_ids, int B,
                                    int pending, int32_t* target_ids, uint16_t* feats, void* stream);

/* Row-wise argmax of bf16 logits (lowest index on ties): the target's greedy
 * ids that dflash_verify consumes. Stateless.
 *  logits device [rows, cols] bf16 (row pitch = cols); out device [rows] int32.
 * Errors: EINVAL (rows < 0, cols < 1, null pointer when rows > 0). */
dflash_status dflash_rows_argmax_bf16(const uint16_t* logits, int rows, int cols,
                                      int32_t* out, void* stream);

/* Wait for all work on the device, then report and clear the context's
 * device status word: OK, ETIMEOUT or EDEVICE. */
dflash_status dflash_sync(dflash_ctx* ctx);

/* ---- temperature sampling and lossless rejection-sampling verify ----
 * The DFlash notes evaluate at temperature 1 ("DFlash - Block Diffusion for
 * Flash Speculative Decoding", 6.2 "Sampling (Temperature = 1)", with the
 * "Lossless Guarantee"; the "DFlash 2" notes at temperature 1, top-p 0.95,
 * top-k 20, lossless rejection sampling). A filtered distribution keeps the
 * top_k largest logits (lower id first among equal logits), takes their
 * softmax at the temperature, keeps the shortest prefix (in that order) whose
 * mass reaches top_p, and renormalises. Lists are DFLASH_SAMPLE_WIDTH wide:
 * ids in decreasing probability, then -1 with probability 0. Draws are
 * inverse-CDF draws with caller-supplied uniforms in [0, 1): the first list
 * entry whose cumulative probability exceeds u. Arguments: temperature > 0,
 * top_k in [1, 32], top_p in (0, 1]; EINVAL otherwise. */
#define DFLASH_SAMPLE_WIDTH 32

/* The drafter pass of dflash_draft with a sampling head: every masked
 * position j is drawn from the drafter's filtered distribution q_j.
 *  uniforms   device [n_seq, B-1] fp32, one per masked position
 *  draft_ids  device [n_seq, B-1] int32 output (the draws)
 *  q_ids      device [n_seq, B-1, 32] int32 output, q_probs fp32 output:
 *             the lists q_j the draws came from (dflash_verify_sample's input)
 * The first call allocates the fp32 logits rows (max_batch*max_block rows of
 * V+256 floats) and the list scratch. Errors: EINVAL (also while a path
 * selector is installed, or vocab above 524288), ENOMEM. */
dflash_status dflash_draft_sample(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq,
                                  const int32_t* anchor_ids, int B, float temperature, int top_k,
                                  float top_p, const float* uniforms, int32_t* draft_ids,
                                  int32_t* q_ids, float* q_probs, void* stream);

/* Filtered distributions of bf16 logit rows (the target's block logits):
 *  logits     device [rows, cols] bf16, row pitch cols, 16-byte aligned;
 *             cols a multiple of 8, 32 <= cols <= 524288; rows <= max_batch*max_block
 *  out_ids    device [rows, 32] int32, out_probs device [rows, 32] fp32
 *  uniforms, drawn  device [rows] fp32 / int32, or both NULL: one draw per row
 * Uses the context's list scratch only (no sequence state). Errors: EINVAL, ENOMEM. */
dflash_status dflash_sample_filter(dflash_ctx* ctx, const uint16_t* logits, int rows, int cols,
                                   float temperature, int top_k, float top_p, const float* uniforms,
                                   int32_t* out_ids, float* out_probs, int32_t* drawn, void* stream);

/* Lossless speculative-sampling verify and commit. Per sequence, walking
 * j = 0..B-2: draft x_j (drawn from q_j) is accepted when
 * u_accept[j] < min(1, p_j(x_j) / q_j(x_j)); at the first rejection the
 * emitted token is drawn from max(0, p_j - q_j) (over p_j's list, in its
 * order) with u_resample[j], tau = j + 1; when every draft is accepted,
 * tau = B and the bonus is drawn from p_{B-1} with u_resample[B-1]. Then the
 * first min(tau, pending) pending tokens are committed, as dflash_verify.
 *  draft_ids, q_ids, q_probs   device, as dflash_draft_sample wrote them
 *  p_ids, p_probs    device [n_seq, B, 32]: the target's filtered lists after
 *                    each block position (dflash_sample_filter of its logits)
 *  u_accept [n_seq, B-1], u_resample [n_seq, B]  device fp32 uniforms
 *  tau, bonus        device [n_seq] int32 outputs
 * Errors: EINVAL. An empty target list latches EDEVICE (reported by sync). */
dflash_status dflash_verify_sample(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, int B,
                                   const int32_t* draft_ids, const int32_t* q_ids, const float* q_probs,
                                   const int32_t* p_ids, const float* p_probs, const float* u_accept,
                                   const float* u_resample, int32_t* tau, int32_t* bonus, void* stream);

/* ---- dynamic block-size scheduling (host logic) ----
 * The DFlash notes (6.5, block size) find that a drafter trained at block 16
 * also serves block 8, which allows choosing B per cycle. The scheduler keeps,
 * per draft position j, exponentially decayed counts of cycles that reached
 * j and that accepted it, read from acceptance lengths tau (tau - 1 leading
 * drafts accepted). Each position's rate is shrunk toward the pooled rate of
 * all positions (positions never reached inherit it): with
 * w = prior_accept + prior_reject,
 * pooled = (sum accepted + prior_accept) / (sum reached + w) and
 * a_j = (accepted_j + w * pooled) / (reached_j + w),
 *     E[tau | B] = 1 + sum_{j=1}^{B-1} prod_{i<=j} a_i,
 * and dflash_block_sched_choose returns, among the sizes whose cycle cost is
 * set, the one with the largest E[tau | B] / cost(B) (the smaller on ties; the
 * smallest size when no cost is set). Host memory only; no CUDA call. */
typedef struct dflash_block_sched dflash_block_sched;

/* sizes: host [n_sizes] distinct block sizes in [1, 32]; decay in (0, 1]
 * (1 = plain counts); priors > 0. Errors: EINVAL, ENOMEM. */
dflash_status dflash_block_sched_create(const int32_t* sizes, int n_sizes, float decay, float prior_accept,
                                        float prior_reject, dflash_block_sched** out);
dflash_status dflash_block_sched_destroy(dflash_block_sched* s);

/* Record n cycles run with block B: taus host [n], each in [1, B]. Errors: EINVAL. */
dflash_status dflash_block_sched_observe(dflash_block_sched* s, int B, const int32_t* taus, int n);

/* Cycle cost of size B (one of the sizes), any positive unit (ms). Errors: EINVAL. */
dflash_status dflash_block_sched_set_cost(dflash_block_sched* s, int B, float cycle_ms);

/* E[tau | B] under the current counts, B in [1, largest size]. Errors: EINVAL. */
dflash_status dflash_block_sched_expected_tau(const dflash_block_sched* s, int B, double* out);

/* The size to run next. Errors: EINVAL. */
dflash_status dflash_block_sched_choose(const dflash_block_sched* s, int* B_out);

/* Install (or remove) the DFlash 2 path selector ("DFlash 2" notes,
 * "Solution - Lightweight Path Selector"). While installed, dflash_draft
 * keeps the 16 largest logits of every masked position t as its candidates
 * C_t (largest first, lower id first among equal logits), scores every
 * adjacent pair a in C_{t-1}, b in C_t as
 *     S_t(a, b) = U_t(b) + < A(a) * H(h_t), B(b) >
 * (U_t the drafter's logit, * elementwise, C_0's predecessor the anchor) and
 * returns the greedy walk: at each position the candidate with the largest
 * score after the previous pick (the higher-ranked one among equal scores),
 * instead of the plain argmax ids. The maps are linear:
 *     A(a) = W_A E[a],  B(b) = W_B E[b],  H(h_t) = W_H h~_t,
 * E the drafter's token embedding and h~_t the final-normalised hidden state
 * that the LM head reads.
 *
 *  w_a, w_b, w_h  device [dim, H] bf16, 16-byte aligned; all three NULL
 *                 removes the selector. W_A and W_B are read only here (the
 *                 library keeps A and B of every token, V x 512 fp32); W_H is
 *                 borrowed like the other weights.
 *  dim            256
 * Enqueued on `stream`, then waits for it. The first install allocates the
 * tables and buffers (V*2 KB plus max_batch*max_block rows of (V+256) fp32
 * logits). Errors: EINVAL (dim != 256, vocab < 16, some but not all pointers
 * NULL, misaligned pointer, vocab above 524288), ENOMEM, ECUDA. */
dflash_status dflash_set_path_selector(dflash_ctx* ctx, const uint16_t* w_a, const uint16_t* w_b,
                                       const uint16_t* w_h, int dim, void* stream);

/* One site of the DFlash 2 two-tap dynamic convolution ("DFlash 2" notes,
 * "Solution - Two-Tap Dynamic Convolution"): over the block positions t of
 * each sequence,
 *     Conv(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}     (* elementwise),
 *     k_{t,i}   = base_i + U_i (V_i x_t),
 * x_{-1} = 0 for the block's first position (the anchor); the first masked
 * position reads the anchor. The correction is a rank-`rank` map of the
 * position's own input (the notes leave its form open; 20 sites of two such
 * taps at rank 80 and hidden 2560 give the 16.5M parameters they state).
 * All three device arrays are bf16, 16-byte aligned, and borrowed like the
 * model weights:
 *   base  [2][hidden]          tap 0 (position t), tap 1 (position t - 1)
 *   u     [2][hidden][rank]
 *   v     [2][rank][hidden] */
typedef struct {
  const uint16_t* base;
  const uint16_t* u;
  const uint16_t* v;
} dflash_conv_site;

/* Install (or remove) the two-tap convolutions of a drafter context: four
 * sites per layer, in the order
 *     ai  on the attention input       h = Conv_ai(RMSNorm(x))
 *     ao  on the attention output      x += Conv_ao(Attn(h) W_o^T)
 *     fi  on the feed-forward input    h = Conv_fi(RMSNorm(x))
 *     fo  on the feed-forward output   x += Conv_fo(FFN(h))
 * `sites` is a host array of 4 * n_layers entries (layer-major); NULL
 * removes the convolutions. The injected context K/V do not pass through
 * them. The library keeps, per layer, V_ao W_o and V_fo W_d (the output
 * sites' products come out of the O and down projections as 2 * rank extra
 * rows) and V_ai, V_fi transposed: 2 * rank * (2 * hidden + n_q * d + ffn)
 * bf16 per layer, plus row buffers for max_batch * max_block rows.
 * While installed, each output site adds the next input site's products
 * over its columns with float atomics, so repeated drafts agree only up to
 * the order of those sums (the plain pass is bit-reproducible).
 * Enqueued on `stream`, then waits for it. Errors: EINVAL (target context,
 * rank not a multiple of 8 in [8, 128], hidden not a multiple of 128, a NULL
 * or misaligned pointer), ENOMEM, ECUDA. */
dflash_status dflash_set_conv(dflash_ctx* ctx, const dflash_conv_site* sites, int rank, void* stream);

/* ---- inspection hooks (used by the parity tests; they synchronise) ---- */

/* Copy `n` cached tokens of layer `layer` of `seq`, starting at position
 * `pos0`, to host buffers k_out / v_out, each [n, n_kv_heads, d] bf16
 * (kv_format 1: the decoded values code * scale, rounded to bf16).
 * Positions may reach into the pending tokens. */
dflash_status dflash_debug_read_kv(dflash_ctx* ctx, int layer, int seq, int pos0, int n,
                                   uint16_t* k_out, uint16_t* v_out);

/* kv_format 1 only: the stored 8-bit blocks of `n` cached tokens, host
 * outputs (any may be NULL): k_codes, v_codes [n, n_kv_heads, d] int8;
 * k_scales, v_scales [n, n_kv_heads, d/32] fp16 bit patterns.
 * EINVAL for a bf16 cache. */
dflash_status dflash_debug_read_kv_q8(dflash_ctx* ctx, int layer, int seq, int pos0, int n, int8_t* k_codes,
                                      uint16_t* k_scales, int8_t* v_codes, uint16_t* v_scales);

/* State of the last dflash_draft call: the final residual stream
 * [n_seq*B, H] fp32 (before the final RMSNorm), and the winning logit of each
 * draft row [n_seq*(B-1)] fp32. Host outputs; either may be NULL. */
dflash_status dflash_debug_last_draft(dflash_ctx* ctx, float* hidden_out, float* top_logit_out);

/* Failure-path check: launches one kernel whose bounded mbarrier wait nothing
 * satisfies; it gives up after limit_us microseconds (1 .. 2e6) and latches the
 * timeout bit, so the next dflash_sync returns DFLASH_ETIMEOUT (and clears it).
 * No fault, no trap; the context stays usable. Errors: EINVAL, ECUDA. */
dflash_status dflash_debug_wait_timeout(dflash_ctx* ctx, int limit_us, void* stream);

/* Selector state of the last dflash_draft call made with the selector
 * installed, per draft row r = i*(B-1) + t (host outputs, any may be NULL):
 *  cand_out    [rows, 16] int32  candidate ids C_t, largest logit first
 *  u_out       [rows, 16] fp32   their logits U_t
 *  scores_out  [rows, 16, 16] fp32  S_t(a, b), a the rank in C_{t-1}, b the
 *              rank in C_t; at t = 0 only a = 0 (the anchor) is defined.
 * EINVAL when the last draft did not run the selector. */
dflash_status dflash_debug_last_selection(dflash_ctx* ctx, int32_t* cand_out, float* u_out, float* scores_out);

/* Y[M, N] (fp32) = X[M, K] * W[N, K]^T with the library's tensor-core GEMM,
 * all device pointers (W, X bf16; K multiple of 8). splits = split-K factor
 * (0 = library's choice). For kernel-level tests. */
dflash_status dflash_debug_gemm(const uint16_t* W, const uint16_t* X, float* Y,
                                int N, int M, int K, int splits, void* stream);

/* Y[M, N] (fp32) = X[M, K] * W[N, K]^T, like dflash_debug_gemm, but without
 * allocating any device memory. The pages have no counterpart: this serves
 * callers that cannot call cudaMalloc, e.g. a loop that must not risk the
 * implicit device synchronisation of cudaMalloc/cudaFree, a process whose
 * free device memory is held by a caching allocator, or code running while
 * another thread has a global-mode stream capture in progress.
 * The split-K workspace, tile tickets and status word live in one fixed
 * 8 MiB + 16 KiB device array inside the library, which every GPU that loads
 * the library holds until the process exits. The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress); make that
 * first call before starting any stream capture. Every call shares the
 * array: the tickets and status are cleared at the start of each call, and
 * calls that overlap on the GPU (other threads or streams) race on it.
 * The call waits for its stream before returning (the status word is read
 * back on that stream; the legacy default stream is not touched unless it is
 * the stream passed).
 * W, X, Y: device pointers (W, X bf16, 16-byte aligned; K a multiple of 8).
 * splits: split-K factor, 0 = chosen to fit the array.
 * Errors: EINVAL for bad arguments, more than 4096 output tiles, or an
 * explicit `splits` above 1 whose partial tiles exceed the fixed scratch
 * (2 x splits x roundup(M, T) x roundup(N, 128) floats above 2^21, T the
 * token tile: 16, 32, 64, 128 or 256, the smallest of these that holds M, and
 * 256 above 128); ECUDA;
 * ETIMEOUT/EDEVICE as reported by the kernel. Messages via
 * dflash_last_error(NULL). */
dflash_status dflash_gemm_noalloc(const uint16_t* W, const uint16_t* X, float* Y,
                                  int N, int M, int K, int splits, void* stream);

/* ---- per-kernel accounting (used by the benchmark) ----
 * Every kernel launch of a context is counted in one of these classes. While
 * profiling is enabled, each launch is also bracketed by two CUDA events
 * recorded on the launch stream, and the algorithmic bytes and flops of the
 * launch (what the operation must read, write and compute; not including
 * split-K or attention partials) are accumulated. */
enum {
  DFLASH_K_QKV = 0,       /* q/k/v projection + RoPE                    */
  DFLASH_K_ATTN,          /* block attention over context chunks        */
  DFLASH_K_ATTN_COMBINE,  /* merge of the attention chunks              */
  DFLASH_K_O,             /* output projection + residual               */
  DFLASH_K_GATEUP,        /* gate/up projection + SwiGLU                */
  DFLASH_K_DOWN,          /* down projection + residual                 */
  DFLASH_K_LMHEAD,        /* LM head + argmax                           */
  DFLASH_K_FUSE_WC,       /* fusion projection W_c                      */
  DFLASH_K_FUSE_KV,       /* context K/V projection + RoPE + append     */
  DFLASH_K_NORM,          /* embedding and RMSNorm rows                 */
  DFLASH_K_VERIFY,        /* verify + commit                            */
  DFLASH_K_OTHER,         /* bookkeeping kernels                        */
  DFLASH_K_SELECT,        /* path selector: top-16, pair scores, walk   */
  DFLASH_K_SAMPLE,        /* top-32 lists, filter and draw              */
  DFLASH_K_CONV,          /* two-tap convolutions (apply kernels)       */
  DFLASH_K_COUNT
};

typedef struct {
  long long launches; /* kernels launched                                 */
  double ms;          /* summed event-timed duration (profiling enabled)  */
  double bytes;       /* summed algorithmic bytes                          */
  double flops;       /* summed algorithmic flops                          */
} dflash_kernel_stat;

/* Enable (1) or disable (0) event timing of every launch of ctx. Counts and
 * algorithmic totals are kept in either case. */
dflash_status dflash_debug_profile(dflash_ctx* ctx, int enable);

/* Synchronise, copy min(n, DFLASH_K_COUNT) class totals to `out` (host), and
 * reset the totals. */
dflash_status dflash_debug_profile_read(dflash_ctx* ctx, dflash_kernel_stat* out, int n);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
