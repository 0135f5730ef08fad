/*
 * bd.h -- C ABI of libbd: the hot path of block-causal masked-diffusion decoding
 * on one GB300 (sm_103a).
 *
 * One denoising step over the active blocks of a block-causal masked-diffusion
 * decoder is made of four calls:
 *
 *   bd_block_causal_attn   attention of the active blocks over the cached prefix
 *   bd_unmask_step         argmax / confidence over the vocabulary and the commit rule
 *   bd_spec_verify         scaffold-speculative verification of a drafted block
 *   bd_fork_rollouts       attention of N rollouts that share one prefix KV cache
 *
 * Conventions shared by every call
 * --------------------------------
 * - Ownership: every data pointer is a caller-owned DEVICE buffer (for example a
 *   torch tensor's data_ptr()).  The library never allocates, frees or keeps a
 *   pointer past the call; all work is enqueued asynchronously on `stream`
 *   (a cudaStream_t, NULL = legacy default stream).
 * - Layout: tensors are dense, row-major in the order their shape is written,
 *   and start on a 16-byte boundary.
 * - Workspace: calls that need scratch memory take a caller-owned device buffer
 *   of at least bd_*_workspace_size(args) bytes.  It must be zero-filled before
 *   its first use; the counter words sit at fixed offsets at its start and every
 *   call that completes leaves them at zero again, so the buffer can be reused
 *   by later calls of any shape on the same stream without clearing.  Calls that
 *   share a workspace must not overlap in time.
 * - Errors: argument errors are found on the host before anything is enqueued
 *   and returned as a bd_status; nothing is launched in that case.  Errors the
 *   device finds (a bounded wait that expired, an inconsistent block partition)
 *   are OR-ed into the optional `dev_status` word (device int32, may be NULL);
 *   bd_check() reads and maps it.
 * - Bounded waits: no kernel waits forever.  Each wait of a kernel's pipeline
 *   (a tile or a piece of logits that has not landed, a stage not yet freed)
 *   gives up after `wait_limit_ns` nanoseconds (0 -> 1 s), sets BD_DEV_TIMEOUT
 *   in *dev_status and makes the call's results invalid; the kernel still lets
 *   every copy and MMA it has issued land (those drains keep the 1 s limit)
 *   and exits, so the stream and context stay usable.  A small limit is a way
 *   to exercise that path.
 * - The kernels are built for sm_103a only; on any other device the calls
 *   return BD_ERR_UNSUPPORTED.
 *
 * Position states, block states and dtypes are the integer constants below.
 */
#ifndef BD_H
#define BD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bd_status {
  BD_OK = 0,
  BD_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes        */
  BD_ERR_UNSUPPORTED = 2,   /* head dim, GQA ratio, alignment or device not supported  */
  BD_ERR_WORKSPACE = 3,     /* workspace missing or smaller than bd_*_workspace_size   */
  BD_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed                       */
  BD_ERR_TIMEOUT = 5,       /* (bd_check) a device-side bounded wait expired           */
  BD_ERR_DEVICE_INPUT = 6   /* (bd_check) the device found an inconsistent input       */
} bd_status;

/* bits OR-ed into *dev_status by the kernels */
#define BD_DEV_TIMEOUT 0x1
#define BD_DEV_BAD_INPUT 0x2

/* per-position state (uint8) */
#define BD_MASKED 0
#define BD_COMMITTED 1
#define BD_SCAFFOLD 2

/* per-block activation status (int32), see bd_unmask_step */
#define BD_INACTIVE 0
#define BD_HALF 1
#define BD_FULL 2
#define BD_DONE 3

/* logits element types; K/V element types (kv_dtype) */
#define BD_F32 0
#define BD_BF16 1
#define BD_E4M3 2

/* -----------------------------------------------------------------------------
 * FP8 KV cache (kv_dtype = BD_E4M3).
 *
 * No counterpart on the pages (their low-precision work concerns weights): a
 * storage variant of the attention operator that halves the K/V bytes read.
 * K and V hold 8-bit floats in the OCP E4M3 format (1 sign, 4 exponent bits
 * of bias 7, 3 mantissa bits; largest value 448), with one power-of-two scale
 * per (KV head, block of 128 rows of the buffer, counted from its first row):
 * the dequantised row r of head h is the E4M3 value times 2^exp[h, r / 128].
 * Exponents must lie in [-15, 7] -- every dequantised value is then exact in
 * fp16 -- and a kernel that meets another one records BD_DEV_BAD_INPUT and
 * uses the nearest bound.  The attention is the computation of the bf16
 * operator over the dequantised cache: the kernel dequantises each tile to
 * fp16 in shared memory and multiplies in fp16 (queries are converted to
 * fp16, exact for 2^-17 <= |q| < 65504).  RoPE and the streaming mask are not
 * supported with E4M3 (BD_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------------*/

/* -----------------------------------------------------------------------------
 * RoPE applied inside the attention operator to pre-RoPE cached keys.
 *
 * FlashDrive tutorial (agifrontier.github.io), section "流式推理": cached keys are
 * kept without position encoding and RoPE is injected in the operator at the
 * re-based position p - Δ after the window slides.
 *
 * With enabled != 0, cached prefix key s is rotated at position k_pos[s] - delta
 * before Q·Kᵀ, rotate-half over the pairs (d, d + D/2) with frequency
 * theta^(-2d/D).  The rotated key enters the bf16 product as the bf16 rounding
 * (to nearest, ties to even) of the rotation formed in float64 -- angle
 * (k_pos[s] - delta) * f_d, then a cos - b sin and b cos + a sin -- exactly,
 * element by element, for |k_pos[s] - delta| < 2^24.  Queries and
 * the active positions' own keys must already be rotated by the caller.  The
 * cache itself is never modified: the call rotates the prefix keys once into
 * its workspace (Hkv * C * D * 2 bytes more, counted by bd_*_workspace_size)
 * and every row tile reads that copy.
 *   k_pos  device int32 [C], or NULL for k_pos[s] = s
 * ---------------------------------------------------------------------------*/
typedef struct bd_rope {
  int32_t enabled;
  const int32_t* k_pos;
  int32_t delta;
  float theta;
} bd_rope;

/* -----------------------------------------------------------------------------
 * bd_block_causal_attn
 *
 * Fast-dVLA paper notes (papernotes.org), "关键设计 1. 分块因果注意力"; Fast-dDrive
 * method summary (e.mffb.com.cn) §3.1; WAM-Diff2 write-up (163.com) §2.1: the
 * output is cut into blocks; a block attends to the whole cached prefix, to every
 * earlier block and bidirectionally to itself, never to a later block.  Block
 * size 1 is ordinary causal attention.
 *
 * For active position i in block b(i), query head h (KV head h / (Hq/Hkv)):
 *   key j is visible  <=>  j < C  or  block(j - C) <= b(i)
 *   o[i, h]   = softmax_j(q[i,h]·k[h',j] · sm_scale) · v[h', j]   (bf16 out)
 *   lse[h, i] = ln Σ_visible exp(q[i,h]·k[h',j] · sm_scale)       (fp32)
 *
 *   q            bf16 [n_q, Hq, D]
 *   k, v         bf16 [Hkv, kv_stride, D]; rows [0, C) cached prefix, rows
 *                [C, C + n_q) the active positions (already rotated); rows past
 *                C + n_q are never read
 *   o            bf16 [n_q, Hq, D]
 *   lse          fp32 [Hq, n_q] natural log, or NULL
 *   block_start  device int32 [n_blocks + 1]: 0 = block_start[0] < ... <
 *                block_start[n_blocks] = n_q; or NULL for uniform blocks of
 *                block_size positions (the last one ragged)
 *   sm_scale     0 -> D^-1/2
 *   num_splits   KV splits (1..16): the CTAs of one thread-block cluster, whose
 *                partial rows meet in the workspace (in L2); 0 -> chosen by the
 *                library, which may also run the call as two launches (whole
 *                waves of unsplit row tiles, then the rest split wide).  With
 *                one split and no RoPE no workspace is needed (NULL is fine)
 *   prefix_ready 0, or 1 to declare that the cached prefix rows [0, C) of k and v
 *                were complete before the kernel that precedes this call on
 *                `stream` started (true of a decode step's KV cache, which the
 *                previous kernel -- the QKV projection of this layer -- does not
 *                write).  The call may then start fetching those rows while
 *                that kernel is still running (programmatic dependent launch);
 *                q, the active rows and every output are touched only after it
 *                has completed.  Ignored with RoPE.
 *   q_pos        NULL, or device int32 [n_q] for the streaming mask (FlashDrive
 *                tutorial, "流式推理": the new frame's tokens are queries over the
 *                cached window, causally in the view-major positions).  Then
 *                the queries attend to the cached rows [0, C) only -- the new
 *                frame's own keys are among them, written by bd_stream_insert
 *                -- and key j is visible to query i iff
 *                pos(j) - rope.delta <= q_pos[i], pos(j) = rope.k_pos[j] (j when
 *                k_pos is NULL), whether or not RoPE is enabled.  block_start /
 *                block_size are ignored; kv_stride >= C suffices.  A query that
 *                sees no key gets o = 0 and lse = -inf.
 * Supported: D in {64, 128}; Hq % Hkv == 0; 1 <= n_q; 0 <= C; kv_stride >= C + n_q.
 * ---------------------------------------------------------------------------*/
typedef struct bd_attn_args {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const int32_t* block_start;
  int32_t n_blocks;
  int32_t block_size;
  int32_t C;
  int32_t n_q;
  int32_t Hq;
  int32_t Hkv;
  int32_t D;
  int32_t kv_stride;
  float sm_scale;
  bd_rope rope;
  int32_t num_splits;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  int32_t prefix_ready;
  const int32_t* q_pos;
  uint64_t wait_limit_ns;
  /* 0 or BD_BF16: k, v bf16.  BD_E4M3: k, v E4M3 bytes [Hkv, kv_stride, D]
   * with exponents k_exp, v_exp int8 [Hkv, ceil(kv_stride / 128)] (device) */
  int32_t kv_dtype;
  const int8_t* k_exp;
  const int8_t* v_exp;
} bd_attn_args;

bd_status bd_block_causal_attn(const bd_attn_args* a, void* stream);
size_t bd_attn_workspace_size(const bd_attn_args* a);

/* -----------------------------------------------------------------------------
 * bd_fork_rollouts
 *
 * Fast-dDrive method summary (e.mffb.com.cn) §3.3 "共享前缀多轨迹Rollout": the
 * first sections are decoded once; their KV cache is shared by N trajectory
 * rollouts, which are forked from it and differ only in their trajectory part.
 *
 * Rollout r's active query i (block b(i)) attends to the whole shared prefix
 * (never copied), to its own private rows [0, priv_len) (its earlier trajectory
 * blocks) and block-causally to its active rows [priv_len, priv_len + n_q).
 *
 *   q                 bf16 [N, n_q, Hq, D]
 *   prefix_k/v        bf16 [Hkv, prefix_stride, D], rows [0, C) used; read only
 *   priv_k/v          bf16 [N, Hkv, priv_stride, D], rows [0, priv_len + n_q) used
 *   o                 bf16 [N, n_q, Hq, D]
 *   lse               fp32 [N, Hq, n_q] or NULL
 *   block_start, n_blocks, block_size, sm_scale, rope, num_splits, prefix_ready:
 *   as in bd_attn_args (rope and prefix_ready concern the shared prefix only)
 * ---------------------------------------------------------------------------*/
typedef struct bd_fork_args {
  int32_t N;
  const void* q;
  const void* prefix_k;
  const void* prefix_v;
  int32_t prefix_stride;
  const void* priv_k;
  const void* priv_v;
  int32_t priv_stride;
  int32_t priv_len;
  void* o;
  float* lse;
  const int32_t* block_start;
  int32_t n_blocks;
  int32_t block_size;
  int32_t C;
  int32_t n_q;
  int32_t Hq;
  int32_t Hkv;
  int32_t D;
  float sm_scale;
  bd_rope rope;
  int32_t num_splits;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  int32_t prefix_ready;
  uint64_t wait_limit_ns;
  /* 0 or BD_BF16: bf16.  BD_E4M3: prefix_k/v and priv_k/v hold E4M3 bytes with
   * exponents prefix_k_exp, prefix_v_exp int8 [Hkv, ceil(prefix_stride / 128)]
   * and priv_k_exp, priv_v_exp int8 [N, Hkv, ceil(priv_stride / 128)] */
  int32_t kv_dtype;
  const int8_t* prefix_k_exp;
  const int8_t* prefix_v_exp;
  const int8_t* priv_k_exp;
  const int8_t* priv_v_exp;
} bd_fork_args;

bd_status bd_fork_rollouts(const bd_fork_args* a, void* stream);
size_t bd_fork_workspace_size(const bd_fork_args* a);

/* -----------------------------------------------------------------------------
 * bd_stream_insert
 *
 * FlashDrive tutorial (agifrontier.github.io), "流式推理": each control step
 * encodes only the newest camera frame; the history frames' K/V stay in the
 * cache, which is laid out view-major (all frames of one camera, then the
 * next), and the new frame's tokens are written into each view's own frame
 * slot -- not appended at the end -- as pre-RoPE keys.
 *
 * The window holds `frames` frame slots of `per_frame` tokens for each of
 * `views` cameras: slot s of view w is cache rows [(w * frames + s) * per_frame,
 * + per_frame).  The call writes the new frame into slot `slot` (the caller's
 * ring index of the oldest frame) of every view, and its positions into k_pos:
 *   k_cache[h, (w*frames + slot)*per_frame + t, :] = new_k[w*per_frame + t, h, :]
 *   v_cache likewise;  k_pos[(w*frames + slot)*per_frame + t] = new_pos[w*per_frame + t]
 * Keys are copied bit for bit (pre-RoPE; attention rotates them at k_pos - delta).
 *
 *   k_cache, v_cache  bf16 [Hkv, cache_stride, D], rows [0, views*frames*per_frame)
 *   k_pos             device int32 [views * frames * per_frame], updated
 *   new_k, new_v      bf16 [views * per_frame, Hkv, D] (the new frame's tokens,
 *                     view by view, as the projection writes them)
 *   new_pos           device int32 [views * per_frame]
 * Supported: D in {64, 128}; 0 <= slot < frames; cache_stride >= views*frames*per_frame.
 * ---------------------------------------------------------------------------*/
typedef struct bd_stream_insert_args {
  void* k_cache;
  void* v_cache;
  int32_t* k_pos;
  const void* new_k;
  const void* new_v;
  const int32_t* new_pos;
  int32_t views;
  int32_t frames;
  int32_t per_frame;
  int32_t slot;
  int32_t Hkv;
  int32_t D;
  int32_t cache_stride;
} bd_stream_insert_args;

bd_status bd_stream_insert(const bd_stream_insert_args* a, void* stream);

/* -----------------------------------------------------------------------------
 * bd_rope_keys
 *
 * FlashDrive tutorial (agifrontier.github.io), "流式推理": RoPE applied to the
 * pre-RoPE cached keys at the re-based position p - Δ.  The rotation that
 * bd_block_causal_attn / bd_fork_rollouts apply inside the call (bd_rope),
 * written out: key s of head h is rotated at k_pos[s] - delta into out[h, s, :],
 * each element the bf16 rounding of the rotation formed in float64.  One
 * rotation then serves every attention pass over the same prefix -- the MDM
 * and AR passes of a speculative round -- which read `out` with RoPE off.
 *
 *   k       bf16 [Hkv, k_stride, D] pre-RoPE keys, rows [0, C) rotated
 *   out     bf16 [Hkv, C, D] (caller-owned; must not overlap k)
 *   rope    k_pos (device int32 [C] or NULL), delta, theta; `enabled` is ignored
 * Supported: D in {64, 128}; |k_pos[s] - delta| < 2^24.
 * ---------------------------------------------------------------------------*/
typedef struct bd_rope_keys_args {
  const void* k;
  int32_t k_stride;
  void* out;
  int32_t Hkv;
  int32_t C;
  int32_t D;
  bd_rope rope;
} bd_rope_keys_args;

bd_status bd_rope_keys(const bd_rope_keys_args* a, void* stream);

/* -----------------------------------------------------------------------------
 * bd_unmask_step
 *
 * Fast-dDrive method summary (e.mffb.com.cn) §3.1 (masked positions predicted
 * by the reverse process), §3.2 mode 2 step 1 (scaffold auto-accepted);
 * Fast-dVLA paper notes, "关键设计 2" (unmasked tokens stay fixed) and "关键设计
 * 4. 流水线并行解码" (half / full activation by the predecessor's completion
 * ratio; confidence threshold; at least a fraction of the remaining tokens).
 *
 * For every candidate position p (state[p] == BD_MASKED and logit_row[p] >= 0):
 *   pred[p] = argmax_v logits[row, v]           (lowest index on ties)
 *   conf[p] = max softmax probability = 1 / Σ_v exp(l_v - max)
 *   lse[p]  = max + ln Σ_v exp(l_v - max)
 * Block status, from the state at call time:
 *   BD_DONE if the block has no masked position; else block 0 is BD_FULL (its
 *   predecessor lies in the cache); else, with r = non-masked positions of the
 *   previous block (scaffold included) over its size:
 *   r >= act_num/act_den -> BD_FULL, r >= add_num/add_den -> BD_HALF, else
 *   BD_INACTIVE (exact integer comparison).
 * Commits (rem = candidates of the block):
 *   BD_FULL:  {conf >= tau_full} ∪ {the n_min most confident candidates},
 *             n_min = min(rem, max(k_fixed, ceil(rem * min_num / min_den))),
 *             equal confidences ranked by lower position;
 *   BD_HALF:  {conf >= tau_half};  BD_INACTIVE / BD_DONE: nothing.
 * A committed position gets tokens[p] = pred[p], state[p] = BD_COMMITTED,
 * commit[p] = 1.  Scaffold and committed positions never change.
 * With write_draft != 0 every other candidate also gets tokens[p] = pred[p]
 * while it stays BD_MASKED: the MDM draft of the scaffold-speculative round
 * (method summary §3.2 mode 2, step 2: one MDM forward drafts every editable
 * position), ready for bd_spec_verify.
 *
 *   logits        [R, V] of logits_dtype (BD_F32 | BD_BF16), row stride logits_ld
 *                 elements (multiple of 8)
 *   logit_row     int32 [n_pos]: logits row of each position, or -1
 *   block_start   int32 [n_blocks + 1] over the n_pos positions (device)
 *   state         uint8 [n_pos] in/out;  tokens int32 [n_pos] in/out
 *   commit        uint8 [n_pos] out;  n_committed, status int32 [n_blocks] out
 *   pred, conf, lse   int32/fp32/fp32 [n_pos] out, or NULL; non-candidates
 *                 get -1 / 0 / 0
 * Supported: n_pos <= 2048 and every block <= 1024 positions.
 * ---------------------------------------------------------------------------*/
typedef struct bd_unmask_args {
  const void* logits;
  int32_t logits_dtype;
  int64_t logits_ld;
  int32_t R;
  int32_t V;
  const int32_t* logit_row;
  int32_t n_pos;
  const int32_t* block_start;
  int32_t n_blocks;
  uint8_t* state;
  int32_t* tokens;
  float tau_full;
  float tau_half;
  int32_t min_num, min_den;
  int32_t k_fixed;
  int32_t add_num, add_den;
  int32_t act_num, act_den;
  uint8_t* commit;
  int32_t* n_committed;
  int32_t* status;
  int32_t* pred;
  float* conf;
  float* lse;
  int32_t write_draft;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  uint64_t wait_limit_ns;
} bd_unmask_args;

bd_status bd_unmask_step(const bd_unmask_args* a, void* stream);
size_t bd_unmask_workspace_size(const bd_unmask_args* a);

/* -----------------------------------------------------------------------------
 * bd_unmask_step_noalloc
 *
 * No counterpart in the paper: a deployment convenience.  Same computation,
 * arguments and results as bd_unmask_step, for callers that cannot allocate
 * device memory -- for example an in-vehicle runtime whose memory plan is fixed
 * at start-up and forbids device allocation afterwards, or a plug-in host that
 * owns all device memory and hands a plug-in only its input and output buffers.
 * Such a caller cannot provide a workspace; this entry point ignores
 * a->workspace / a->workspace_bytes and uses a scratch array of
 * BD_UNMASK_NOALLOC_SCRATCH_BYTES inside the library instead (every GPU that
 * loads the library holds it until the process exits).  It allocates nothing.
 *
 * - Problems needing more scratch than that (bd_unmask_workspace_size(a) larger
 *   than BD_UNMASK_NOALLOC_SCRATCH_BYTES) are refused with BD_ERR_WORKSPACE.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - Each call clears the array's counter words on `stream` first; the rest of
 *   the array keeps the previous call's contents.
 * - All calls share the one array: calls whose work overlaps on the GPU (other
 *   streams, or no ordering between them) race and give wrong results.
 * ---------------------------------------------------------------------------*/
#define BD_UNMASK_NOALLOC_SCRATCH_BYTES (1u << 20)
bd_status bd_unmask_step_noalloc(const bd_unmask_args* a, void* stream);

/* -----------------------------------------------------------------------------
 * bd_spec_verify
 *
 * Fast-dDrive method summary (e.mffb.com.cn) §3.2 "模式二：Scaffold Speculative
 * Decoding": scaffold accepted as is; the MDM draft of the block's editable
 * positions is compared left to right with the AR argmax; matches are accepted;
 * at the first mismatch the AR token is taken, later drafts are dropped, and a
 * bonus token is accepted.  Fast-dDrive abstract / §1: for test-time scaling the
 * AR verifier of the trajectory section is sampled.
 *
 * For each sequence s of n_seq (independent rollouts), with E = number of
 * non-scaffold slots of its block and e the editable ordinal of a slot:
 *   t_e = argmax_v ar[s, e, v]                       (greedy, noise == NULL)
 *   t_e = argmax_v (ar[s,e,v] / temperature - ln(-ln u[s,e,v]))   (sampled)
 * Going over the masked editable slots in order (committed slots are skipped):
 * a slot whose draft equals t_e is committed; the first one that differs takes
 * t_e, is committed and is the bonus; masked slots after it return to masked
 * with token -1.  If none differs, the bonus is t_E (row E), which belongs to
 * the position after the block (bonus_pos = L).
 *
 *   tokens        int32 [n_seq, L] in/out (masked slots hold the draft)
 *   state         uint8 [n_seq, L] in/out
 *   ar_logits     [n_seq, n_rows, V] of logits_dtype, row stride logits_ld;
 *                 n_rows must equal E + 1 for every sequence
 *   noise         fp32 [n_seq, n_rows, V] uniforms in (0, 1), row stride
 *                 logits_ld, or NULL for greedy
 *   accepted_len  int32 [n_seq] out: slots committed this round, bonus included
 *   bonus, bonus_pos  int32 [n_seq] out
 * Supported: L <= 1024, n_seq <= 1024, n_seq * n_rows <= 65535.
 * ---------------------------------------------------------------------------*/
typedef struct bd_verify_args {
  int32_t n_seq;
  int32_t L;
  int32_t* tokens;
  uint8_t* state;
  const void* ar_logits;
  int32_t logits_dtype;
  int64_t logits_ld;
  int32_t n_rows;
  int32_t V;
  const float* noise;
  float temperature;
  int32_t* accepted_len;
  int32_t* bonus;
  int32_t* bonus_pos;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  uint64_t wait_limit_ns;
} bd_verify_args;

bd_status bd_spec_verify(const bd_verify_args* a, void* stream);
size_t bd_verify_workspace_size(const bd_verify_args* a);

/* -----------------------------------------------------------------------------
 * Helpers
 * ---------------------------------------------------------------------------*/
const char* bd_status_string(bd_status s);

/* Synchronises `stream`, reads *dev_status and maps its bits: BD_DEV_TIMEOUT ->
 * BD_ERR_TIMEOUT, BD_DEV_BAD_INPUT -> BD_ERR_DEVICE_INPUT, 0 -> BD_OK.  The word
 * is left as it is (clear it with cudaMemsetAsync to reuse it). */
bd_status bd_check(const int32_t* dev_status, void* stream);

/* Library version, "major.minor.patch". */
const char* bd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BD_H */
