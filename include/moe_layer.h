/*
 * moe_layer.h -- C ABI of the block-quantized MoE layer library (sm_103a).
 *
 * One sparse MoE FFN layer as the Step-5 / Step-3.7 pages describe it
 * ("Step-5 Preview GGUF", "Model background" table: hidden 4096, 352 routed
 * experts, 8 selected per token, shared experts; "Precision distribution"
 * table and "Step 3.7 Flash Mixed-Quant GGUF", "Tensor recipe" table: routed
 * experts in low-bit block types such as Q4_K, shared experts in Q8_0, the
 * router in F32), run on the small token batch of MTP verification
 * ("Support Step3.5/3.7 flash mtp3", llama.cpp PR #24340, "Overview",
 * Round 1 step 1: [id_last, d1, d2, d3], all logits on), plus the greedy
 * acceptance of that PR's steps 4 and 5.
 *
 * Layer definition (the pages name the tensors but print no formula; this is
 * the plain reading the library implements):
 *   l[t,e] = sum_h x[t,h] Wr[e,h] + b[e];  p = softmax_e(l[t,:]);
 *   ids[t,0..k-1] = the k largest p (descending, ties to the lower e);
 *   g[t,j] = p[t,ids[t,j]] / sum_j' p[t,ids[t,j']];
 *   FFN_e(v) = Wd_e (silu(Wg_e v) * (Wu_e v)),  silu(u) = u / (1 + e^-u);
 *   y[t] = sum_j g[t,j] FFN_ids[t,j](x[t]) + FFN_shared(x[t]).
 *
 * Arithmetic:
 *   - T <= 8: weights enter as their integer codes; x and the SwiGLU outputs
 *     as 32-value block fixed point (16-bit limbs in bf16 mode, 32-bit in
 *     fp32 mode).  Every block product is therefore exact, and block sums are
 *     scaled and accumulated in fp32.
 *   - The router logits are fp32 sums over 512-column slices, added across
 *     slices and to the bias exactly (as integer multiples of 2^-32) and
 *     rounded once.
 *   - The same inputs give the same output bits on every call.
 *   - T > 8: weights are dequantised to bf16; bf16 tensor-core products with
 *     fp32 accumulation.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless a comment says "host".
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  The caller owns every buffer it passes.
 *   - Return value: MOE_OK or a negative MOE_E* code.  On error nothing is
 *     launched unless the code is MOE_ECUDA; moe_last_error() then describes
 *     the failure.  No call aborts or throws.
 *   - Arguments are validated on the host before anything touches the GPU.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_EINVAL (-1)   /* bad argument (null, size, alignment, T out of range) */
#define MOE_ENOMEM (-2)   /* device allocation failed */
#define MOE_EFORMAT (-3)  /* unsupported format, or a shape the format cannot hold */
#define MOE_ETIMEOUT (-4) /* a bounded device-side wait gave up (see moe_layer_status) */
#define MOE_ECUDA (-5)    /* a CUDA runtime call failed */

/* Weight formats.  Serialised layouts (blocks run along a row, i.e. along
 * the reduction dimension K = cols):
 *   MOE_F32  : row-major fp32.
 *   MOE_Q8_0 : 32 weights -> 34 bytes: fp16 d (little endian), 32 x int8 q;
 *              w = d * q.  The pages name Q8_0 without a layout; this is the
 *              library's reading of it.
 *   MOE_Q4KS : the library's Q4_K-style type.  256 weights -> 144 bytes:
 *              fp16 d, fp16 dmin, sixteen 6-bit fields (sc[0..7], m[0..7]) as
 *              one little-endian bit stream in 12 bytes, then 128 bytes of
 *              4-bit codes (weight i in byte 16 + i/2, low nibble for even i);
 *              w = (d*sc[s]) * q - dmin*m[s] for sub-block s = i/32.
 *   MOE_BF16 : reserved (not accepted for weights). */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_Q8_0 = 2, MOE_Q4KS = 3 } moe_fmt;

/* Activation / output type of moe_forward.
 *   MOE_ACT_BF16: x and y are bf16.  Inside, x and the SwiGLU outputs enter
 *                 the integer dot products as 16-bit block fixed point
 *                 (per 32 values: a power-of-two scale and 16-bit integers).
 *   MOE_ACT_F32 : "check mode": x and y are fp32, block fixed point has 32
 *                 bits.  Slower; meant for verification. */
typedef enum { MOE_ACT_BF16 = 0, MOE_ACT_F32 = 1 } moe_act;

/* A serialised weight matrix [rows, cols].  `data` may be a host or a device
 * pointer; it is read only during moe_layer_create. */
typedef struct {
  int32_t fmt;      /* moe_fmt */
  int32_t reserved; /* must be 0 */
  int64_t rows, cols;
  const void* data;
  size_t nbytes; /* must equal moe_quantized_bytes(fmt, rows, cols) */
} moe_tensor;

typedef struct {
  int32_t H;         /* hidden size; multiple of 256 */
  int32_t E;         /* routed experts, 1..1024 */
  int32_t top_k;     /* experts per token, 1..min(E, 16) */
  int32_t I;         /* routed expert intermediate size; multiple of 32 (256 for MOE_Q4KS) */
  int32_t I_shared;  /* shared expert intermediate size; 0 = no shared expert */
  int32_t T_max;     /* largest token count moe_forward will be given, 1..8192 */
  int32_t act_dtype; /* moe_act */
  uint32_t wait_limit_us; /* bound of every device-side wait, in microseconds
                             (0 = the default, 2 s); a wait that runs out ends
                             the launch with MOE_ETIMEOUT (moe_layer_status) */
  moe_tensor router_w; /* [E, H], MOE_F32 */
  moe_tensor router_b; /* [1, E], MOE_F32; data == NULL for no bias */
  const moe_tensor* gate; /* HOST array of n descriptors, each [I, H] */
  const moe_tensor* up;   /* HOST array of n descriptors, each [I, H] */
  const moe_tensor* down; /* HOST array of n descriptors, each [H, I] */
  moe_tensor sh_gate, sh_up, sh_down; /* [I_shared, H], [I_shared, H], [H, I_shared];
                                         the format may differ from the routed one */
  /* Expert parallelism: the layer may hold only the routed experts
   * [expert_begin, expert_begin + n) of the E the router scores, n =
   * expert_count (0 = all E, with expert_begin 0); gate/up/down then describe
   * those n experts in order.  Such a layer routes every token over all E
   * experts (the router is replicated) and its forward returns that shard's
   * part of y: sum over the token's chosen experts that it holds of
   * g[t,j] FFN(x[t]), plus the shared expert if it has one (I_shared > 0).
   * The sum of the parts of shards that cover every expert once, with the
   * shared expert on exactly one of them, is the layer's y (residual: give
   * exactly one shard moe_forward_residual). */
  int32_t expert_begin;
  int32_t expert_count;
} moe_layer_desc;

typedef struct moe_layer moe_layer;

/* Uploads and repacks every weight into the library's device layout and
 * allocates all workspace, on the current device.  The caller may free the
 * source buffers once the call returns (it synchronises `stream`).
 * Errors: MOE_EINVAL (null pointers, sizes), MOE_EFORMAT (format/shape),
 * MOE_ENOMEM, MOE_ECUDA.  *out is set only on success. */
int moe_layer_create(const moe_layer_desc* desc, void* stream, moe_layer** out);

/* y[T, H] = MoE(x[T, H]) for 0 <= T <= T_max, in the layer's act_dtype.
 * x and y must be 16-byte aligned and must not overlap.  T == 0 returns
 * MOE_OK and launches nothing.  No allocation happens here.  Calls on one
 * layer must not run concurrently (they share the layer's workspace).
 * Device-side wait failures are reported by moe_layer_status().
 * Launch overlap (T <= 8): the kernel is launched with programmatic stream
 * serialization.  Its blocks may start while the previous kernel in the
 * stream is still running; before that kernel completes they only read the
 * layer's own constant weights, and they wait for it (and for its memory
 * operations) before reading x or the workspace.  Stream order is therefore
 * kept for every kernel, whether or not the previous kernel triggers early.
 * The kernel lets the next kernel in the stream launch early too. */
int moe_forward(moe_layer* L, const void* x, int32_t T, void* y, void* stream);

/* y = x + MoE(x): a residual layer (the target stack of an MTP round,
 * "Support Step3.5/3.7 flash mtp3", "Overview" step 2).  Same arguments,
 * rules and errors as moe_forward; the sum is formed in fp32 and rounded
 * once to the act_dtype. */
int moe_forward_residual(moe_layer* L, const void* x, int32_t T, void* y, void* stream);

/* y = MoE(x) as fp32 [T, H] whatever the layer's act_dtype, for callers that
 * keep the residual stream in fp32 (as the pages' runtime keeps its hidden
 * states in F32 tensors, "Support Step3.5/3.7 flash mtp3", "Overview"): the
 * combine's fp32 sum is stored without the rounding to bf16.  T <= 8 only
 * (MOE_EINVAL above); otherwise the arguments, rules and errors of
 * moe_forward, with y (4 T H bytes) 16-byte aligned and not overlapping x. */
int moe_forward_f32(moe_layer* L, const void* x, int32_t T, float* y, void* stream);

/* One pre-norm residual block's step of the residual stream, in the layer's
 * own launch ("Support Step3.5/3.7 flash mtp3", "Overview": the target
 * stack keeps F32 hidden states; the pre-norm residual reading of the block
 * is this library's, h <- h + MoE(rmsnorm(h))):
 *   h_out = h_in + MoE(x)                       (fp32 [T, H])
 *   xn    = h_out / sqrt(mean(h_out^2) + eps)   (act dtype [T, H], weight 1)
 * x [T, H] (act dtype) is the block's input, normally the previous step's
 * xn.  The mean over the H columns of a row is summed per 128-column block
 * and then over the blocks in order (fp32, deterministic).  Nothing is
 * written to a y; the routing and the status are those of moe_forward.
 *   0 <= T <= min(8, T_max); h_in, h_out, xn 16-byte aligned; h_in == h_out
 *   (in place) or not overlapping it; x, xn, h_out pairwise disjoint, and xn
 *   disjoint from h_in; eps finite and >= 0.  Asynchronous, no allocation.
 * Errors: MOE_EINVAL (arguments), MOE_ECUDA. */
int moe_forward_resnorm(moe_layer* L, const void* x, int32_t T, const float* h_in, float* h_out, void* xn, float eps,
                        void* stream);

/* Copies the routing of the last moe_forward (device-to-device, async on
 * `stream`): ids int32 [T, k] and gates fp32 [T, k] in slot order, offsets
 * int32 [E+1], perm int32 [T*k] (pair ids t*k+j grouped by expert, ascending
 * within an expert).  Any pointer may be NULL to skip it.  The stream
 * argument orders the copies after the forward on the caller's stream, so
 * reading the routing never synchronises the device. */
int moe_get_routing(moe_layer* L, int32_t* ids, float* gates, int32_t* offsets, int32_t* perm,
                    void* stream);

/* Synchronises `stream` and reads the layer's device status word: MOE_OK, or
 * MOE_ETIMEOUT if a bounded device-side wait gave up in some earlier call
 * (the word is then cleared and the workspace re-zeroed). */
int moe_layer_status(moe_layer* L, void* stream);

/* Phase timeline of the layer's last completed T <= 8 launch, for
 * profiling: synchronises `stream`, then writes n (>= 1) int64 values to the
 * HOST array out_ns, in nanoseconds of the GPU's global timer relative to
 * the first of the launch's blocks to pass its dependency wait, -1 where the
 * event did not happen.  The events, in order:
 *   0 first block entered the kernel (before its dependency wait; negative
 *     when it started during the previous kernel)
 *   1 first block passed its dependency wait (0 by definition)
 *   2 the activation records of x were complete (written by the router
 *     tiles: the same time as 3)
 *   3 the last router tile finished (the routing starts)
 *   4 the routing was published
 *   5 first routed gate/up weight copy issued
 *   6 first routed gate/up stage computed
 *   7 the shared expert's gate/up outputs were complete
 *   8 the last routed entry's gate/up outputs were complete
 *   9 first routed down weight copy issued
 *  10 the last block found the work queue exhausted
 *  11 the last 128-row block of the down outputs was complete
 *  12 the last combine finished
 *  13 first block leaving
 *  14 last block leaving
 *  15 the last combining block started its combine
 *  16 the last combining block had the routing arrays it needs
 *  17 the routing's top-k and gates were done
 *  18 the routing's permutation and work entries were written
 * (-1 for i >= 19).  The stamps cost a few atomic writes per block and are
 * always recorded. */
int moe_layer_timeline(moe_layer* L, int64_t* out_ns, int32_t n, void* stream);

/* Test hook for the bounded device-side waits (no fault is involved).
 * site 1: the layer's next T <= 8 forward waits for a routing publication
 * that never comes (its work-claiming threads wait for a flag value the
 * kernel does not write).  That wait runs out after the layer's
 * wait_limit_us, every other thread of the launch sees the status word and
 * stops, all copies in flight are drained, and moe_layer_status() then
 * returns MOE_ETIMEOUT naming the "routing flag" site and clears the state;
 * later forwards are unaffected.  The output of the failed forward is
 * undefined.  Other sites: MOE_EINVAL. */
int moe_layer_inject_timeout(moe_layer* L, int32_t site);

/* Bytes of weights resident on the device (repacked), and of workspace. */
size_t moe_layer_weight_bytes(const moe_layer* L);
size_t moe_layer_workspace_bytes(const moe_layer* L);

void moe_layer_destroy(moe_layer* L);

/* Serialised size of a [rows, cols] matrix in `fmt`; 0 if the shape does not
 * fit the format. */
size_t moe_quantized_bytes(int32_t fmt, int64_t rows, int64_t cols);

/* Quantises fp32 w [rows, cols] (device) into serialised `fmt` bytes at out
 * (device, moe_quantized_bytes(...) bytes).  MOE_Q8_0: d = max|w|/127 in
 * fp32, stored as fp16; q = clamp(round_half_away(w / d), -127, 127).
 * MOE_Q4KS: the closed-form min/max quantiser (per sub-block A = (hi - lo)/15
 * with lo = min(0, min w), B = -lo; d, dmin = fp16(max A / 63), fp16(max B / 63);
 * sc, m = round(A / d), round(B / dmin) clamped to [0, 63];
 * q = clamp(round((w + dmin*m) / (d*sc)), 0, 15)).  Bit-exact and
 * deterministic. */
int moe_quantize(int32_t fmt, const float* w, int64_t rows, int64_t cols, void* out, void* stream);

/* Greedy verification of k drafted tokens against the target's logits over
 * the verify batch ("Support Step3.5/3.7 flash mtp3", "Overview", Round 1
 * steps 4-5): a_i = argmax_v logits[i, v] (ties to the lowest v) for
 * i = 0..k; *out_n_accepted = the largest n <= k with a_i == draft_ids[i]
 * for all i < n; *out_next_token = a_n (the correction token, or the bonus
 * token when all drafts match).  The caller hands pending_h =
 * verify_h[*out_n_accepted] to the next round.
 *   draft_ids int32 [k] (device), logits fp32 [k+1, V] row-major (device,
 *   finite values), outputs int32 (device).  0 <= k <= 15, 1 <= V <= 2^24.
 *   workspace: device scratch of mtp_verify_accept_workspace_bytes(k, V)
 *   bytes, 16-byte aligned, owned by the caller; it must be zero-filled
 *   before its first use and is left zero-filled by every call that
 *   completes.  Calls sharing one workspace must not overlap on the GPU.
 *   The scratch is the caller's rather than the library's so that the call
 *   never allocates (it stays capturable in a CUDA graph) and calls on
 *   different workspaces may run concurrently; mtp_verify_accept_noalloc
 *   below takes no workspace.
 *   Launched with programmatic stream serialization like moe_forward: it
 *   waits for the previous kernel in the stream before reading anything. */
size_t mtp_verify_accept_workspace_bytes(int32_t k, int32_t V);
int mtp_verify_accept(const int32_t* draft_ids, int32_t k, const float* logits, int32_t V,
                      int32_t* out_n_accepted, int32_t* out_next_token, void* workspace,
                      size_t workspace_bytes, void* stream);

/* The same greedy verification as mtp_verify_accept, for callers that cannot
 * allocate device memory: a C runtime driving the draft/verify loop without a
 * device allocator of its own, for which cudaMalloc / cudaFree would also
 * synchronise the device between verify rounds.  The source pages have no
 * counterpart to this call; it only changes where the scratch lives.
 *   Arguments, outputs and results are those of mtp_verify_accept; the
 *   scratch is a 4096-byte array inside the library (one per device), so
 *   the call accepts only 16 + 8 * (k+1) * ceil(V / 16384) <= 4096 (every
 *   V <= 507904 for every k <= 15) and returns MOE_EINVAL, with a message
 *   naming the sizes, beyond that.  It allocates nothing and calls no
 *   allocating library.  Every call looks the array's device address up in
 *   the current context (so a call after cudaDeviceReset finds the array of
 *   the new context); the first call on a device also loads the library's
 *   module there, so make it before any stream capture on that device.
 *   The array keeps the last call's contents: its first 16 bytes (a
 *   counter) are zero at module load and every completed call leaves them
 *   zero; the rest is written before it is read.  All calls on a device
 *   share the array: calls whose kernels overlap on the GPU (different
 *   streams, other host threads) race and must be ordered by the caller,
 *   e.g. by issuing them on one stream. */
int mtp_verify_accept_noalloc(const int32_t* draft_ids, int32_t k, const float* logits, int32_t V,
                              int32_t* out_n_accepted, int32_t* out_next_token, void* stream);

/* ------------------------------------------------------------------------
 * Output head and one MTP draft/verify round.
 * ------------------------------------------------------------------------ */
typedef struct moe_lm_head moe_lm_head;

/* Uploads a Q8_0 output matrix w [V, H] ("Step-5 Preview GGUF", "Precision
 * distribution" table: the main output matrix is Q8_0); `w.data` may be a
 * host or device pointer and is read only during the call (which
 * synchronises `stream`).  1 <= V <= 2^24, H a positive multiple of 512 and
 * at most 16384, 1 <= T_max <= 8.  act_dtype (moe_act) is the type of the
 * rows forward() is given.  Errors: MOE_EINVAL, MOE_EFORMAT (w not Q8_0 or
 * wrong shape), MOE_ENOMEM, MOE_ECUDA. */
int moe_lm_head_create(const moe_tensor* w, int32_t T_max, int32_t act_dtype, void* stream, moe_lm_head** out);

/* logits fp32 [T, V] = w . rmsnorm(x) for x [T, H] in the head's act_dtype,
 * rmsnorm(v) = v / sqrt(mean(v^2) + eps) (weight 1; the output norm before
 * the LM head).  0 <= T <= T_max; x 16-byte aligned; asynchronous. */
int moe_lm_head_forward(moe_lm_head* lm, const void* x, int32_t T, float eps, float* logits, void* stream);
/* Synchronises `stream` and reports MOE_ETIMEOUT if a bounded device-side
 * wait of an earlier moe_lm_head_forward (or of an mtp_round's LM-head
 * passes) gave up (the word is then cleared); MOE_OK otherwise. */
int moe_lm_head_status(moe_lm_head* lm, void* stream);
void moe_lm_head_destroy(moe_lm_head* lm);

/* One MTP draft/verify round on synthetic weights, the reading of
 * "Support Step3.5/3.7 flash mtp3", "Overview" steps 1-6 used by this
 * library (the pages give the data flow, not a synthetic model):
 *   h_0 = x (the verify batch [k+1, H]); h_{l+1} = h_l + MoE_l(rmsnorm(h_l))
 *   for the n_target layers (pre-norm residual blocks); logits = lm(h_n)
 *   (output norm + LM head), written to target_logits fp32 [k+1, V];
 *   head j (j < k) runs on rmsnorm of the j+1 rows h~_j = h_n[0..j] +
 *   noise[j][0..j] (the noise stands in for an imperfect draft model) and
 *   writes head_out[j] ([k][k][H], rows 0..j used; may be NULL to discard);
 *   draft_ids[j] = argmax (lowest id on ties) of lm(h~_j[j]), whose logits
 *   go to draft_logits fp32 [k, V] (may be NULL to discard);
 *   draft confidence cut ("Step-3.5-Flash MTP GGUF", "Usage":
 *   --spec-draft-p-min, 0.65 recommended; 0 in the PR's runs): p_j = the
 *   softmax probability of draft j's token under its logits (fp32,
 *   1 / sum_v exp(l_v - max l)); drafting stops at the first j with
 *   p_j < p_min, and draft_ids[j..k-1] are set to -1 (p_min = 0 keeps
 *   every draft);
 *   then greedy acceptance as mtp_verify_accept over the kept drafts.
 * The residual stream h and the noisy rows h~ are kept in fp32 in both
 * act dtypes: the target layers' inputs rmsnorm(h) are in act_dtype, and
 * each layer adds its output to h in fp32 and normalises the next layer's
 * input in its own launch (moe_forward_resnorm); head outputs are in
 * act_dtype.
 * Every layer and the head must share act_dtype; all layers have hidden H,
 * T_max >= k+1.  noise fp32 [k][k][H] (device).  1 <= k <= 7.
 * workspace: device scratch of mtp_round_workspace_bytes(H, k, V, act)
 * bytes, 256-byte aligned, zero-filled before its first use and left so.
 * Asynchronous; no allocation.  Errors: MOE_EINVAL on any mismatch, or
 * p_min < 0 / NaN. */
size_t mtp_round_workspace_bytes(int32_t H, int32_t k, int32_t V, int32_t act_dtype);
int mtp_round(moe_layer* const* target_layers, int32_t n_target, moe_layer* const* draft_heads, int32_t k,
              moe_lm_head* lm, const void* x, const float* noise, float eps, float p_min, void* workspace,
              size_t workspace_bytes, float* target_logits, float* draft_logits, void* head_out, int32_t* draft_ids,
              int32_t* out_n_accepted, int32_t* out_next_token, void* stream);

/* Copies the final residual rows h_n (fp32 [k+1, H], the LM head's input for
 * the verify rows, and with the noise the source of the draft rows) of the
 * last mtp_round that ran on `workspace` with these H, k, V, act_dtype and
 * n_target into h_out (device, fp32 [k+1, H]).  The round leaves them in its
 * workspace; this reads them for checking the round's last steps (output
 * norm, LM head, drafts, acceptance) on their own.  Ordered on `stream`
 * after the round when the round used the same stream.  Errors: MOE_EINVAL
 * (NULL pointer, n_target < 0, sizes outside mtp_round_workspace_bytes'
 * ranges, workspace too small), MOE_ECUDA. */
int mtp_round_hidden(const void* workspace, size_t workspace_bytes, int32_t H, int32_t k, int32_t V, int32_t act_dtype,
                     int32_t n_target, float* h_out, void* stream);

/* Message for the last error on the calling thread; valid until the next
 * call on that thread.  Never NULL. */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LAYER_H */
