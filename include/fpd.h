/*
 * fpd.h — C ABI of the GB300 (sm_103a) block-drafter hot path.
 *
 * One non-causal block drafter pass of diffusion-drafter speculative decoding, the per-position
 * constrained argmax over legal vocabulary slices, and the acceptance-length scan.  The method:
 *
 *   - VFlash paper (Chinese translation), §2.1 "Preliminaries": features of selected target layers are
 *     fused and injected as keys and values into every drafter layer; given the start token the drafter
 *     predicts the masked positions of a block in ONE bidirectional forward pass; greedy verification
 *     accepts up to the first position that disagrees with the target.
 *   - VFlash blog, "Method": text runs in verified-SD mode with 16-position blocks (one accepted anchor +
 *     15 proposals); the target keeps the longest matching prefix plus its own next token.
 *   - VFlash paper (zh), §2.2: a block of length L is one observed start token followed by L-1 masked
 *     tokens, all predicted conditionally independently in one pass.
 *   - VFlash paper (zh), §2.3: coordinates use one of 1001 dedicated tokens, or a fixed-width field of one
 *     sign slot and five digit slots whose unused high digits are filled with a mask token.
 *   - VFlash paper (zh), §2.5 "Inference": per-position constraints restrict coordinates and delimiters to
 *     their legal vocabulary, acting on already-computed logits; a primitive is accepted when its schema
 *     validator passes, otherwise the first k draft positions are retained.
 *   - FlashDrive, §3.2 "Diffusion-based drafting": the drafter conditions on fused target hidden states
 *     written into the draft layers' KV cache and produces a whole candidate block in one pass.
 *
 * Conventions (all entry points):
 *   - Every tensor argument is memory the CALLER owns (device memory unless marked "host").  The library
 *     never frees caller memory.  Weights are borrowed and must outlive the model handle.
 *   - Element types: bf16 for activations/weights/KV (passed as void*), int32 ids, fp32 logits.
 *   - Layouts are row-major.  Weight matrices are [out_features, in_features].
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy default stream).
 *     No call synchronises, allocates device memory, or copies host<->device.  Every call validates its
 *     arguments on the host first and returns an error WITHOUT launching anything when they are wrong.
 *   - Errors: a non-zero fpd_status; fpd_last_error() returns a message for the calling thread.
 *     FPD_ERR_CUDA wraps a CUDA runtime error seen at launch.
 *   - Device pointers passed to the library must be 16-byte aligned.
 */
#ifndef FPD_H_
#define FPD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FPD_MAX_LAYERS 8
#define FPD_MAX_CLASSES 32   /* vocabulary classes in one layout */
#define FPD_MAX_RANGES 64    /* [lo,hi) id ranges over all classes of one layout */
#define FPD_MAX_PAIRS 128    /* cross-position pairs of one layout */

typedef enum {
  FPD_OK = 0,
  FPD_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, misaligned pointer */
  FPD_ERR_SHAPE = 2,         /* inconsistent or unsupported sizes */
  FPD_ERR_CAPACITY = 3,      /* workspace / KV store / position table too small, table limits exceeded */
  FPD_ERR_UNSUPPORTED = 4,   /* model shape the kernels do not implement */
  FPD_ERR_CUDA = 5,          /* CUDA runtime/driver error at launch */
  FPD_ERR_DEVICE_CHECK = 6   /* a kernel reported a failed device-side check (see fpd_device_status) */
} fpd_status;

/* Codes of the device-side check word (fpd_device_status): the first failure a kernel recorded.  Kernels never
 * trap; they record the code and skip or clamp the offending access. */
enum {
  FPD_CHECK_BAD_TOKEN = 1,      /* an id outside [0, V) reached the embedding gather (row zeroed) */
  FPD_CHECK_WAIT_TIMEOUT = 2,   /* an mbarrier / flag wait exceeded its 1 s limit (the kernel abandoned its loop) */
  FPD_CHECK_NO_LEGAL_ID = 3,    /* a position's vocabulary class admits no id (token -1) */
  FPD_CHECK_BAD_CLASS = 4,      /* a pos_class entry outside [0, n_class) */
  FPD_CHECK_BAD_CONTEXT = 5,    /* a ctx_len outside [0, t_cap] (clamped) */
  FPD_CHECK_BAD_POSITION = 6,   /* a context row's position pos_start[b] + i outside [0, t_cap) (row skipped) */
  FPD_CHECK_CTX_OVERFLOW = 7    /* fpd_sd_advance: ctx_len + accepted rows would pass t_cap (rows capped) */
};

/* Drafter shape.  The layer form is a pre-norm transformer layer with per-head q/k RMSNorm, rotate-half
 * RoPE, grouped-query attention without any mask (bidirectional over context + block) and a SwiGLU MLP;
 * an untied LM head follows a final RMSNorm.  Supported: head_dim in {64, 128}; d_model, d_ff multiples of
 * 64; n_q_heads a multiple of n_kv_heads. */
typedef struct fpd_model_desc {
  int32_t n_layers;     /* 1..FPD_MAX_LAYERS (5 for the five-layer drafter) */
  int32_t d_model;      /* d */
  int32_t n_q_heads;    /* H_q */
  int32_t n_kv_heads;   /* H_kv */
  int32_t head_dim;     /* h */
  int32_t d_ff;         /* SwiGLU inner width F */
  int32_t vocab;        /* V */
  int32_t n_feat;       /* number of fused target layers n_f (1..8) */
  int32_t max_pos;      /* RoPE positions [0, max_pos) are supported: context capacity + block length */
  float rms_eps;        /* RMSNorm epsilon: y = x / sqrt(mean(x^2) + eps) * g */
  float rope_theta;     /* RoPE base: angle(pos, i) = pos * theta^(-2i/h), i < h/2 */
} fpd_model_desc;

/* Borrowed device weights, all bf16, row-major [out, in]. */
typedef struct fpd_weights {
  const void* embed;        /* [V, d] token embedding (anchor and mask rows) */
  const void* w_fc;         /* [d, n_f*d] fusion projection over the concatenated target features */
  const void* hidden_norm;  /* [d] RMSNorm gain applied to the fused context */
  const void* final_norm;   /* [d] RMSNorm gain before the LM head */
  const void* lm_head;      /* [V, d] */
  const void* attn_norm[FPD_MAX_LAYERS];  /* [d] */
  const void* wqkv[FPD_MAX_LAYERS];       /* [(H_q + 2 H_kv) h, d]: rows of q heads, then k heads, then v heads */
  const void* q_norm[FPD_MAX_LAYERS];     /* [h] per-head RMSNorm gain on q */
  const void* k_norm[FPD_MAX_LAYERS];     /* [h] per-head RMSNorm gain on k (context and block keys) */
  const void* wo[FPD_MAX_LAYERS];         /* [d, H_q h] */
  const void* mlp_norm[FPD_MAX_LAYERS];   /* [d] */
  const void* w_gate_up[FPD_MAX_LAYERS];  /* [2F, d]: rows 0..F-1 gate, rows F..2F-1 up */
  const void* w_down[FPD_MAX_LAYERS];     /* [d, F] */
} fpd_weights;

typedef struct fpd_model fpd_model;

/* Per-position legal vocabulary (VFlash paper (zh), §2.5: coordinates and delimiters restricted to their
 * legal vocabulary).  Class c is the union of id ranges [lo, hi) listed in
 * class_ranges[2*class_off[c] .. 2*class_off[c+1]).  A class may be the full vocabulary ([0, V)).
 * The tables are HOST memory (they are part of the declared layout and small); pos_class is DEVICE
 * memory, one class id per block position of every request, [B*L] int16 (position 0, the anchor, is
 * ignored).  Ranges of one class must be non-empty, inside [0, V), sorted and disjoint. */
typedef struct fpd_vocab_layout {
  int32_t n_class;               /* 1..FPD_MAX_CLASSES */
  const int32_t* class_off;      /* host [n_class + 1], class_off[0] = 0, total ranges <= FPD_MAX_RANGES */
  const int32_t* class_ranges;   /* host [2 * class_off[n_class]] (lo, hi) pairs */
  const int16_t* pos_class;      /* device [B * L] */
  /* Cross-position rule (f3; VFlash paper (zh) §2.5: a cross-position rule pairs off-screen coordinates, acting on
   * the computed logits).  For every declared pair (p, q) of block positions and every request, both positions
   * take off_id or neither does: with a_x the largest logit of x's legal ids other than off_id and o_x the logit
   * of off_id at x, both take off_id when o_p + o_q > a_p + a_q (fp32 sums), else both take their best other
   * id.  off_id must be legal at both positions.  n_pairs = 0 (zero-initialised struct) disables the rule. */
  int32_t n_pairs;               /* 0..FPD_MAX_PAIRS */
  const int16_t* pairs;          /* host [2 * n_pairs]: (p, q), 1 <= p, q < L, p != q */
  int32_t off_id;
} fpd_vocab_layout;

/* Schema rules for primitive-mode acceptance, one int8 per block position (device [B*L]).
 * VFlash paper (zh), §2.3 and §2.5: the validator checks the declared layout; fixed-width numerals pad
 * only their unused HIGH digits with the mask token, so a field reads [sign][pad..pad][digit..digit]. */
enum {
  FPD_RULE_NONE = 0,        /* not checked */
  FPD_RULE_MEMBER = 1,      /* token must lie in its position's class */
  FPD_RULE_DIGIT = 2,       /* digit slot, not the last of its field: member; pad_id allowed only while the
                               previous slot is not a digit slot holding a real digit */
  FPD_RULE_DIGIT_LAST = 3,  /* last digit slot of a field: member, must be a real digit (!= pad_id), and
                               the same ordering rule as FPD_RULE_DIGIT */
  FPD_RULE_CONFIDENT = 4    /* member, and the drafter's top-2 margin at the position is at least tau
                               (fpd_verify_prefix; fails like a schema rule otherwise) */
};

enum { FPD_VERIFY_TEXT = 0, FPD_VERIFY_SCHEMA = 1 };

/* ---- model handle ------------------------------------------------------------------------------------
 * Validates the shape, records the borrowed weight pointers, and builds the model's own small device
 * tables (the RoPE cos/sin table for max_pos positions and TMA descriptors of the weights).  This is the
 * one call that allocates device memory (those tables); it synchronises the current device once. */
fpd_status fpd_model_create(const fpd_model_desc* desc, const fpd_weights* weights, fpd_model** out);
void fpd_model_destroy(fpd_model* model);

/* ---- f2: 8-bit weights for the weight-streaming calls ----------------------------------------------------------
 * FlashDrive §3.4 "Quantization": low-bit weights cut the bytes a memory-bound decoding step loads, and 8-bit
 * activations let the products run on 8-bit matrix units.  Here both operands of the streamed GEMMs take E4M3
 * (the OCP OFP8 format: bias 7, largest finite 448) with one power-of-two scale per 128 consecutive elements of a
 * row:
 *   exponent k = the smallest integer with amax 2^-k <= 448 (amax: the group's largest magnitude; k clamped to
 *   [-126, 127]; k = 0 for an all-zero group); code = the E4M3 value nearest to x 2^-k, ties to the even code, a
 *   zero result encoded +0; the group stands for decode(code) 2^k.
 *
 * fpd_model_enable_fp8 quantises, once, the model's QKV, O, gate/up and down matrices of every layer and the LM
 * head into a device allocation the model owns (about half the bytes of the bf16 matrices; freed by
 * fpd_model_destroy) and synchronises the stream.  From then on the calls that stream these weights use them:
 *   fpd_draft_block with batch * block_len <= 16, and fpd_constrain_argmax without a layout and with
 *   batch * (block_len - 1) <= 16.
 * In those calls each projection quantises its bf16 input rows the same way (per token, per 128 elements) and
 * computes y = sum over groups of (codes . codes) 2^(k_x + k_w) in fp32.  Every other call (context preparation,
 * larger blocks, constrained LM heads) keeps the bf16 weights.  The borrowed bf16 weights must stay valid.
 * Needs d_model, n_q_heads * head_dim and d_ff to be multiples of 128 (FPD_ERR_UNSUPPORTED otherwise); calling it
 * again is a no-op.  Not capturable in a CUDA graph (it allocates and synchronises). */
fpd_status fpd_model_enable_fp8(fpd_model* model, void* stream);
/* 1 after a successful fpd_model_enable_fp8, else 0. */
int32_t fpd_model_fp8_enabled(const fpd_model* model);

/* The quantisation above on any bf16 matrix, on the device (stream-ordered, asynchronous).
 *   w      device [rows, ld] bf16, 16-byte aligned; cols a positive multiple of 128, ld >= cols and a multiple of 8
 *   codes  device [rows, cols] uint8 E4M3 codes, 16-byte aligned
 *   exps   device [rows, cols / 128] int8 exponents k */
fpd_status fpd_quantize_fp8(const void* w, int rows, int cols, int ld, void* codes, void* exps, void* stream);

/* Bytes of the caller-allocated context KV store for `batch` requests of at most t_cap context positions.
 * Layout: [layer][request][K|V][kv_head][t_cap][head_dim] bf16. */
size_t fpd_kv_store_bytes(const fpd_model* model, int batch, int t_cap);

/* Bytes of caller-allocated scratch ("workspace") that is enough for every call below with these sizes
 * (block_len <= max_block_len, total context rows <= batch * t_cap).  Workspace contents do not survive
 * between calls except where stated (fpd_draft_block writes nothing that later calls read). */
size_t fpd_workspace_bytes(const fpd_model* model, int batch, int max_block_len, int t_cap);

/* ---- a1 + a2: context fusion and per-layer context K/V --------------------------------------------------
 * VFlash paper (zh), §2.1; FlashDrive §3.2.  For each packed context row r of request b:
 *   ctx_r = RMSNorm_{hidden_norm}( [F_0,r | F_1,r | ... | F_{n_f-1},r] . w_fc^T )              (bf16)
 *   for every layer l and kv head g:  K^l_g(pos) = RoPE_pos( RMSNorm_{k_norm[l]}( ctx_r . Wk^l_g^T ) ),
 *                                     V^l_g(pos) = ctx_r . Wv^l_g^T                              (bf16)
 * with pos = pos_start[b] + (r - row_off[b]) (pos_start NULL means 0: a fresh context), written into
 * kv_store at [l][b][K|V][g][pos][:].
 *   feats      host array of n_feat DEVICE pointers, each [total_rows, d] bf16 (rows of all requests packed)
 *   row_off    device [batch + 1], row_off[0] = 0, row_off[batch] = total_rows, non-decreasing
 *   pos_start  device [batch] or NULL; the caller guarantees pos_start[b] + rows_b <= t_cap
 * Rows beyond the written positions are left untouched. */
fpd_status fpd_prepare_context(fpd_model* model, int batch, int total_rows, const int32_t* row_off,
                               const int32_t* pos_start, const void* const* feats, void* kv_store,
                               int t_cap, void* workspace, size_t workspace_bytes, void* stream);

/* The same with per-request row counts, for appends whose sizes are known only on the device (the accepted
 * counts of a speculative step, e.g. in a captured CUDA graph).  Rows [row_off[b], row_off[b] + row_cnt[b]) of
 * request b are written at positions pos_start[b] + i; rows past row_cnt[b] inside [row_off[b], row_off[b+1])
 * and rows past row_off[batch] are read but not written.  Here row_off[batch] <= total_rows (total_rows sizes
 * the launch) and row_cnt[b] <= row_off[b+1] - row_off[b].
 *   row_cnt    device [batch] int32, or NULL for row_off[b+1] - row_off[b] */
fpd_status fpd_prepare_context_rows(fpd_model* model, int batch, int total_rows, const int32_t* row_off,
                                    const int32_t* row_cnt, const int32_t* pos_start, const void* const* feats,
                                    void* kv_store, int t_cap, void* workspace, size_t workspace_bytes, void* stream);

/* ---- a3..a7: one bidirectional drafter pass over a block --------------------------------------------------
 * Block of request b: position 0 holds anchor[b], positions 1..L-1 hold mask_id (VFlash (zh) §2.2).
 * Block position j sits at RoPE position ctx_len[b] + j.  Every layer attends, without a mask, over the
 * request's ctx_len[b] context keys/values of that layer followed by the L block keys/values.
 *   ctx_len       device [batch], 0 <= ctx_len[b] <= t_cap (caller guarantees; kernels clamp and record
 *                 FPD_CHECK_BAD_CONTEXT)
 *   anchor        device [batch] token ids in [0, V)
 *   hidden_out    device [batch * L, d] bf16: residual stream after the last layer (before final norm)
 *   layer_hidden  device [n_layers, batch * L, d] bf16 or NULL: residual stream after every layer */
fpd_status fpd_draft_block(fpd_model* model, int batch, int block_len, const void* kv_store, int t_cap,
                           const int32_t* ctx_len, const int32_t* anchor, int32_t mask_id,
                           void* hidden_out, void* layer_hidden, void* workspace,
                           size_t workspace_bytes, void* stream);

/* ---- a8: final RMSNorm, LM head, per-position legal-vocabulary mask, argmax ------------------------------
 * For block positions j = 1..L-1 of every request: z = RMSNorm_{final_norm}(hidden[b,j]) (bf16), logits
 * over the LEGAL ids of the position's class only (illegal ids are never computed), token = argmax in fp32
 * with the lowest id winning ties.
 *   hidden      device [batch * L, d] bf16 (fpd_draft_block's hidden_out)
 *   layout      NULL: every position may take any id in [0, V)
 *   tokens_out  device [batch, L-1] int32
 *   logits_out  device [batch * (L-1), V] fp32 or NULL; only legal columns are written
 *   margin_out  device [batch * (L-1)] fp32 or NULL: the largest minus the second largest fp32 logit over the
 *               position's legal ids (0 on a tie; +inf when the class has a single legal id).  The margin tells a
 *               caller how close the argmax decision was. */
fpd_status fpd_constrain_argmax(fpd_model* model, int batch, int block_len, const void* hidden,
                                const fpd_vocab_layout* layout, int32_t* tokens_out, float* logits_out,
                                float* margin_out, void* workspace, size_t workspace_bytes, void* stream);

/* ---- a8 without a workspace argument ----------------------------------------------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers that cannot allocate device memory
 * (a host framework that owns the whole device heap and forbids plugins to call cudaMalloc, or a latency-critical
 * loop where cudaMalloc's implicit device synchronisation is not allowed).  It computes exactly what
 * fpd_constrain_argmax computes, with the same arguments minus the workspace: its scratch memory is a fixed
 * 8 MiB array in the library's device memory (present on every device that loads the library until the process
 * exits), so the caller supplies only inputs and outputs.  It has no margin output.
 *   - Limit: batch * (block_len - 1) positions whose scratch fits 8 MiB (about 1300 positions at d_model 2560);
 *     larger calls return FPD_ERR_CAPACITY with a message naming the bytes needed, without launching anything.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture on that device.
 *   - Every call on a device shares the one array.  Calls whose kernels overlap on the GPU (other streams,
 *     other host threads) race on it and give undefined results; serialise them.  Each call resets the parts
 *     of the array it reads before reading them, so nothing carries over from the previous call.
 *   - No call allocates or frees device memory. */
fpd_status fpd_constrain_argmax_noalloc(fpd_model* model, int batch, int block_len, const void* hidden,
                                        const fpd_vocab_layout* layout, int32_t* tokens_out, float* logits_out,
                                        void* stream);

/* ---- a9: acceptance-length scan ----------------------------------------------------------------------------
 * FPD_VERIFY_TEXT (VFlash blog "Method"; VFlash (zh) §2.1): target [B, L] holds t_1..t_L, the target's
 *   greedy token at block positions 1..L (t_L follows the last draft).  n = length of the longest prefix
 *   with draft[b, i-1] == t_i; accept_len = n + 1; committed = d_1..d_n, t_{n+1}.
 * FPD_VERIFY_SCHEMA (VFlash (zh) §2.5): position j = 1..L-1 fails when its rule (FPD_RULE_*) fails; with
 *   p the first failing position, accept_len = p - 1 (all L-1 when none fails); committed = d_1..d_k.
 *   Needs layout (membership) and rule (device [B*L] int8); target is ignored.
 *   draft       device [B, L-1] int32
 *   accept_len  device [B] int32
 *   committed   device [B, L] int32, entries past accept_len set to -1
 *   valid_out   device [B] int32 or NULL: 1 when nothing failed (text: n == L-1) */
fpd_status fpd_verify(int mode, int batch, int block_len, const int32_t* draft, const int32_t* target,
                      const fpd_vocab_layout* layout, const int8_t* rule, int32_t pad_id,
                      int32_t* accept_len, int32_t* committed, int32_t* valid_out, void* stream);

/* ---- f3: primitive acceptance that keeps a prefix up to the first uncertain coordinate ----------------------
 * VFlash paper (zh) §2.5: the prediction passes an acceptance test (the schema validator and, for bounding boxes,
 * a spatial confidence check); the first k draft positions are kept, and for bounding boxes k stops before the
 * first uncertain coordinate.  Reading: a coordinate is uncertain when the drafter's own top-2 logit margin there
 * (fpd_constrain_argmax's margin_out) is below tau.  Position j = 1..L-1 fails when its rule (FPD_RULE_*) fails,
 * FPD_RULE_CONFIDENT also failing when margin[b][j-1] < tau; with p the first failing position, accept_len = p - 1
 * (all L - 1 when none fails), committed = d_1..d_accept, valid = (p == L).
 *   margin  device [B, L-1] float (the margins of the drafted positions); other arguments as fpd_verify's schema
 *           mode */
fpd_status fpd_verify_prefix(int batch, int block_len, const int32_t* draft, const float* margin, float tau,
                             const fpd_vocab_layout* layout, const int8_t* rule, int32_t pad_id, int32_t* accept_len,
                             int32_t* committed, int32_t* valid_out, void* stream);

/* ---- multi-block speculative loop: the step between verification and the next block ----------------------
 * VFlash blog, "Method" (blocks are drafted and verified one after another until the sequence ends);
 * FlashDrive §3.2 (the target's features at the accepted positions extend the drafter's context).  After a
 * text verification of the block [anchor, d_1..d_{L-1}] at positions ctx_len[b] .. ctx_len[b] + L - 1 with
 * accept_len[b] = n + 1 committed tokens (d_1..d_n and the target's token at the first mismatch):
 *   pos_start[b] = ctx_len[b]                     where the target's features of the anchor and the n accepted
 *                                                 draft positions (accept_len[b] rows) are appended
 *   ctx_len[b]  += accept_len[b]                  the next block's context
 *   anchor[b]    = committed[b][accept_len[b] - 1]  the next block's anchor: the last committed token
 * accept_len[b] itself is the row count of that append (fpd_prepare_context_rows row_cnt).  One kernel; no host
 * synchronisation, so a draft -> argmax -> verify -> advance -> append sequence can be captured in a graph.
 * When ctx_len[b] + accept_len[b] would exceed t_cap the count is capped (accept_len[b] is lowered in place),
 * FPD_CHECK_CTX_OVERFLOW is recorded and the anchor is the last committed token that still fits.
 *   accept_len  device [batch] int32 (in/out), committed device [batch, L] int32
 *   ctx_len     device [batch] int32 (in/out), pos_start, anchor device [batch] int32 (out) */
fpd_status fpd_sd_advance(int batch, int block_len, int t_cap, int32_t* accept_len, const int32_t* committed,
                          int32_t* ctx_len, int32_t* pos_start, int32_t* anchor, void* stream);

/* ---- f4: fixed-width grid -> the target's text format (host-side) ----------------------------------------
 * VFlash paper (zh) §2.3: for targets that tokenise numbers as text, every coordinate gets one sign slot and
 * `width` digit slots with unused HIGH digits filled by the mask (pad) token; the grid keeps each position's
 * role and is converted back to the target's text format afterwards, its separators marking block boundaries.
 * Block layout (request b, block position j = 0..L-1; j = 0 is the start token): waypoint w occupies positions
 * 1 + w * (n_axes * (1 + width) + 1) onwards: n_axes fields [sign][d_1..d_width], then one separator.
 * The text of request b is the values of its first complete waypoints among the accepted positions 1..accept[b]
 * (a waypoint counts when all its n_axes fields lie inside the accepted prefix): each field's value as a decimal
 * integer (leading zeros dropped, "-" only for a negative non-zero value), axes joined by axis_sep, waypoints by
 * point_sep.  A field that breaks the schema (a sign slot that is neither plus nor minus, a pad after a real digit,
 * a pad or a non-digit in the last slot) ends the request's text there.
 *   committed  HOST [batch, block_len] int32: fpd_verify's committed tokens (block positions 1..L-1 at 0..L-2)
 *   accept     HOST [batch] int32: accepted positions
 *   out        HOST buffer of out_bytes; request b's NUL-terminated text starts at out + offsets[b]
 *   offsets    HOST [batch + 1]: offsets[batch] = total bytes written (FPD_ERR_CAPACITY when out is too small)
 * Pure host code: needs no GPU. */
typedef struct fpd_grid_format {
  int32_t digit_id[10];   /* token ids of the digits 0..9 */
  int32_t plus_id, minus_id, pad_id;
  int32_t n_axes;         /* fields per waypoint */
  int32_t width;          /* digit slots per field (>= 1) */
  char axis_sep, point_sep;
} fpd_grid_format;

fpd_status fpd_grid_to_text(int batch, int block_len, const int32_t* committed, const int32_t* accept,
                            const fpd_grid_format* fmt, char* out, size_t out_bytes, size_t* offsets);

/* ---- diagnostics ---------------------------------------------------------------------------------------- */
const char* fpd_last_error(void);          /* thread-local message of the last failing call */
uint64_t fpd_kernel_launches(void);        /* kernels launched by this library since load (all threads) */
/* Reads and clears the device-side check word (bounded-wait timeouts, bad ids).  Synchronises the stream.
 * Returns FPD_OK when no kernel recorded a failure, else FPD_ERR_DEVICE_CHECK with *code set. */
fpd_status fpd_device_status(void* stream, int32_t* code);

#ifdef __cplusplus
}
#endif
#endif /* FPD_H_ */
