/*
 * vh.h -- C interface of the GB300 paged q_len=1 decode-attention library.
 *
 * One decode step of a Talker/LM layer for a batch of requests, in three
 * calls on the caller's CUDA stream:
 *
 *   vh_rope_kv_append     RoPE on the new q and k, then append of k and v
 *                         into each request's current KV page;
 *   vh_paged_decode_attn  single-token GQA attention of every request over
 *                         its pages, split across CTAs where a request is
 *                         long, writing finished rows and partial results;
 *   vh_decode_combine     log-sum-exp merge of the partial results.
 *
 * Sources of the operation (pages this library was written from):
 *   - "Engineering TTS inference in vLLM-Omni" (vLLM blog), Fish Speech S2 Pro,
 *     "model-specific attention kernel": decode-only attention with q_len = 1,
 *     bf16, head_dim 128, block size 16, GQA where one kv head serves its
 *     group of q heads; long sequences are split into segments whose partial
 *     max / sum / accumulator are merged by the online-softmax recurrence;
 *     the short/long choice is made without a device-to-host sync.
 *   - same page, Qwen3-TTS section 4 "numerical precision": RoPE cos/sin and
 *     attention are kept in fp32.
 *   - "Adding a Model" (vox-serve docs), "How a program runs": one row per
 *     request, static shapes, no host sync, inputs in device buffers; padding
 *     entries (active == 0) point at the dummy KV page 0, compute garbage
 *     that is ignored and must never write another request's state.
 *   - same page, section "1. The model code": keys and values are written
 *     into the paged cache, then attention runs over it; cache layout
 *     [num_layers, num_pages, 2, page_size, num_kv_heads, head_dim].
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers owned by the caller (except the
 *     step inputs and output that VH_FLAG_HOST_IO lets vh_decode_fused take
 *     in pinned host memory); the library allocates nothing, frees nothing
 *     and keeps no state between calls other than per-device launch settings
 *     it caches on first use (and the fixed scratch array of
 *     vh_paged_decode_attn_noalloc).
 *   - 16-bit values are passed as uint16_t bit patterns: vh_bf16 is always
 *     bf16; vh_e16 is bf16, or IEEE fp16 when the call's flags hold
 *     VH_FLAG_FP16 (the Fish kernel of the first source above takes either
 *     type).  One call uses one type for all of its 16-bit arrays.
 *   - Strides are in ELEMENTS.  One layer's cache is reached through
 *     k_cache / v_cache plus page_stride (elements between pages),
 *     token_stride (elements between token slots of a page) and head_stride
 *     (elements between the kv heads of a slot); element d of head h of slot
 *     t of page n is at n*page_stride + t*token_stride + h*head_stride + d.
 *     Token-major pages [NP, 2, P, Hkv, D] (the vox-serve layout, "NHD"):
 *     v_cache = k_cache + P*Hkv*D, page_stride = 2*P*Hkv*D, token_stride =
 *     Hkv*D, head_stride = D.  Head-major pages [NP, 2, Hkv, P, D] ("HND"):
 *     v_cache = k_cache + Hkv*P*D, page_stride = 2*Hkv*P*D, token_stride = D,
 *     head_stride = P*D.  All three strides must be multiples of 8 elements
 *     (16 bytes); the caller guarantees that distinct (page, slot, head)
 *     rows do not overlap.  Both layouts take the same path: the cache is
 *     described to the copy engine as a 4-D tensor with these strides.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Every call checks its scalar arguments and pointer alignment on the
 *     host, launches asynchronously and never synchronises or reads device
 *     memory on the host, so a sequence of calls can be captured in a CUDA
 *     graph.  Make the first call of each function on a device before any
 *     capture: it sets per-kernel launch attributes once.
 *   - Return value: VH_OK (0) or a negative VH_E* status; a negative status
 *     means nothing was launched, except VH_ECUDA, which reports the CUDA
 *     error raised by the launch itself.
 *   - Data errors found on the device never trap: the offending row is
 *     skipped (or clamped, see below) and a VH_ERR_* bit is ORed into
 *     *err_flag when err_flag is not NULL.  The caller reads it later.
 *
 * Shapes: B rows, Hq q heads, Hkv kv heads (Hq % Hkv == 0, G = Hq / Hkv
 * in {1, 2, 4, 8}), head dim D in {64, 128}, page size 1 <= P <= 1024, a
 * multiple of 16 or exactly 8 when max_pages_per_seq > 1 (with 8-token pages
 * every 16-token tile of the attention spans two pages), 1 <= B <= 65535 and small
 * enough for the attention kernels' shared-memory plan, which keeps 12
 * bytes per row (tile count, length, position) in every CTA: up to about
 * 17,000 rows (fewer kv heads per CTA as B grows); beyond that the calls
 * that plan return VH_EINVAL before any launch.  seq_len
 * counts the token being appended: row b attends over logical slots
 * 0 .. seq_lens[b]-1, and the new token is slot seq_lens[b]-1, i.e. page
 * page_table[b][(L-1)/P], offset (L-1) % P.  page_table is int32
 * [B][max_pages_per_seq], row-major.
 *
 * Contiguous caches: page_table may be NULL; row b's logical page j is then physical page
 * b * max_pages_per_seq + j (B * max_pages_per_seq <= num_pages).  With
 * max_pages_per_seq = 1 and P = the cache length, this is a per-request
 * contiguous cache such as the Fast AR cache of the vLLM-Omni blog's Fish
 * Speech section ("Fast AR buffer reuse": K/V preallocated per layer as
 * [batch][kv head][position][head_dim], one new token written and read in
 * place per step): page_stride = Hkv*P*D, token_stride = D, head_stride =
 * P*D, k_cache and v_cache the layer's two tensors.
 */
#ifndef VH_H
#define VH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t vh_bf16;  /* a bf16 bit pattern */
typedef uint16_t vh_e16;   /* a 16-bit element: bf16, or fp16 under VH_FLAG_FP16 */

/* return codes */
#define VH_OK 0
#define VH_EINVAL (-1)      /* bad shape, NULL pointer or out-of-range scalar */
#define VH_EALIGN (-2)      /* a pointer or stride is not 16-byte aligned */
#define VH_EWORKSPACE (-3)  /* workspace NULL or smaller than required */
#define VH_ECUDA (-4)       /* CUDA reported an error at launch */
#define VH_ENODEV (-5)      /* no usable sm_103 device is current */
#define VH_ESCRATCH (-6)    /* shape needs more scratch than VH_STATIC_SCRATCH_BYTES */

/* device-side data-error bits, ORed into *err_flag */
#define VH_ERR_SEQLEN 1     /* active row with seq_len outside [1, max_pages_per_seq*P]: row skipped */
#define VH_ERR_PAGE 2       /* page id outside [0, num_pages): the append or the page read is skipped */
#define VH_ERR_POS 4        /* position outside [0, max_pos): the row is skipped by the append */
#define VH_ERR_TIMEOUT 8    /* an internal pipeline wait ran out of time: the CTA gave up */

/* flags (the `flags` argument of the calls that take one) */
#define VH_FLAG_PDL 1u      /* programmatic dependent launch (vh_decode_fused, vh_paged_decode_attn) */
#define VH_FLAG_FP16 2u     /* 16-bit elements (q, k_new, v_new, cache, out) are IEEE fp16, not bf16 */
#define VH_FLAG_ROPE_INTERLEAVED 4u /* RoPE pairs elements (2i, 2i+1) instead of (i, i + D/2) */
#define VH_FLAG_PDL_KV 8u   /* VH_FLAG_PDL, and the cached K/V may be requested before the wait (vh_decode_fused) */
#define VH_FLAG_PLANNED 16u /* the workspace holds this step's plan from vh_decode_plan (vh_decode_fused, vh_paged_decode_attn) */
#define VH_FLAG_PLAN_THREE_CALL 32u /* vh_decode_plan: plan for vh_paged_decode_attn instead of vh_decode_fused */
#define VH_FLAG_HOST_IO 64u /* vh_decode_fused: the per-step inputs and out may be pinned host memory, read and written in place */

/* Fill the RoPE table used by vh_rope_kv_append.  Source: "Engineering TTS
 * inference in vLLM-Omni", Qwen3-TTS section 4 (RoPE cos/sin kept in fp32).
 * cos_sin: float [max_pos][D]; row p holds cos(p * f_i) in columns 0..D/2-1
 * and sin(p * f_i) in columns D/2..D-1, f_i = theta^(-2i/D).  Angles and
 * cos/sin are evaluated in double and stored as float (the pages keep RoPE
 * cos/sin in fp32 for alignment with the reference model).  Init-time call.
 * Errors: VH_EINVAL if cos_sin is NULL, max_pos < 1, D not in {64, 128} or
 * theta <= 0; VH_EALIGN if cos_sin is not 16-byte aligned. */
int vh_rope_table(float* cos_sin, int max_pos, int head_dim, double theta, void* stream);

/* RoPE + KV append, one CTA per row.  Sources: "Adding a Model" (vox-serve),
 * section "1. The model code" (RoPE on q and k, then the new key and value
 * written into the paged cache before attention); "Engineering TTS inference
 * in vLLM-Omni", Qwen3-TTS section 4 (RMSNorm variance and RoPE in fp32).
 * q      e16 [B][Hq][D]   new queries (contiguous)
 * k_new  e16 [B][Hkv][D]  new keys, rotated here before they are stored
 * v_new  e16 [B][Hkv][D]  new values, stored bit for bit
 * cos_sin float [max_pos][D] from vh_rope_table
 * positions int32 [B] or NULL; NULL means position = seq_lens[b] - 1
 * q_norm_w, k_norm_w float [D] or NULL: per-head RMSNorm applied to every q
 *        head / new k head before RoPE, x <- w * x / sqrt(mean(x^2) + norm_eps),
 *        in fp32 (the pages keep "RMSNorm variance" in fp32 for alignment);
 *        NULL skips it.  16-byte aligned.  norm_eps >= 0.
 * k_cache, v_cache, page_stride, token_stride, head_stride: the layer's paged cache
 * num_pages: pages in the pool, used only to bounds-check page ids (> 0)
 * page_table int32 [B][max_pages_per_seq], or NULL (contiguous cache, see above);
 *        seq_lens, active int32 [B]
 * q_rot  float [B][Hq][D] out: rotated q in fp32 (rows with active == 0
 *        are not written)
 * err_flag int32* or NULL
 * flags  0 or VH_FLAG_FP16 | VH_FLAG_ROPE_INTERLEAVED
 * For every active row: q_rot = rope(q); the cache slot of token
 * seq_len-1 receives rne(rope(k_new)) (rounded to nearest even in the
 * element type) and v_new.  Rotation is computed in fp32; pair i, at angle
 * pos * theta^(-2i/D), is (i, i + D/2) ("rotate half"), or (2i, 2i + 1)
 * with VH_FLAG_ROPE_INTERLEAVED (the GPT-J pairing).  Rows with
 * active == 0 write nothing.  Precondition (not checked): live rows own
 * disjoint append slots.
 * Errors: VH_EINVAL (NULL pointer other than positions/err_flag/page_table/norm weights, bad shape,
 * max_pos < 1, num_pages < 1, max_pages_per_seq < 1, unknown flags),
 * VH_EALIGN (a pointer or a stride not 16-byte aligned), VH_ECUDA. */
int vh_rope_kv_append(const vh_e16* q, const vh_e16* k_new, const vh_e16* v_new,
                      const float* cos_sin, int max_pos, const int32_t* positions,
                      const float* q_norm_w, const float* k_norm_w, float norm_eps,
                      vh_e16* k_cache, vh_e16* v_cache, int64_t page_stride,
                      int64_t token_stride, int64_t head_stride, int num_pages,
                      const int32_t* page_table, int max_pages_per_seq,
                      const int32_t* seq_lens, const int32_t* active,
                      float* q_rot, int32_t* err_flag, unsigned flags,
                      int B, int Hq, int Hkv, int D, int page_size, void* stream);

/* Number of CTAs per kv-head group that vh_paged_decode_attn launches on the
 * current device when num_ctas == 0 (a multiple of the SM count).  A host
 * helper of this library's split plan (the pages have no counterpart; their
 * kernel picks its split from a CPU upper bound of the length).  Returns a
 * negative VH_E* status on bad shapes or when no device is usable. */
int vh_decode_num_ctas(int B, int Hq, int Hkv, int D, int page_size);

/* Bytes of workspace vh_paged_decode_attn / vh_decode_combine / vh_decode_fused
 * need for this shape and CTA count (num_ctas == 0: enough for the automatic
 * count of either path on the current device).  Returns 0 on bad arguments.
 * A host helper (the pages have no counterpart): the workspace holds the
 * per-segment partial results of the split rows, see vh_decode_combine. */
size_t vh_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size, int num_ctas);

/* Paged GQA decode attention.
 * Source: "Engineering TTS inference in vLLM-Omni", Fish Speech S2 Pro,
 * "model-specific attention kernel": q_len = 1 attention of every request
 * over its cache blocks, one kv head serving its group of q heads, long
 * sequences cut into segments that write partial (max, sum, accumulator)
 * results, the choice made without a device-to-host sync.
 * q_rot float [B][Hq][D] (from vh_rope_kv_append); cache as above.
 * out e16 [B][Hq][D]: rows whose keys one CTA covered entirely are written
 *     here directly; rows with active == 0 (or flagged VH_ERR_SEQLEN) are
 *     written as zeros; rows split across CTAs are finished by
 *     vh_decode_combine.
 * sm_scale: softmax scale; <= 0 means 1/sqrt(D).
 * num_ctas: CTAs per kv-head group, 0 = automatic.  The work is the list of
 *     16-token tiles of all active rows in row order; on the device each CTA
 *     takes an equal contiguous share of that list (no host sync), so a row
 *     is split exactly where its tiles straddle two CTAs.
 * workspace / workspace_bytes: caller-owned device scratch of at least
 *     vh_decode_workspace_bytes(...) bytes, 256-byte aligned; it holds the
 *     per-row split plan and the fp32 partial results.  No initialisation
 *     is needed.  Calls that overlap on the device must use distinct
 *     workspaces.
 * flags: VH_FLAG_FP16 (cache and out are fp16) and VH_FLAG_PDL: launch as a
 *     programmatic dependent of the previous kernel on the stream (for
 *     instance vh_rope_kv_append): lengths, flags and page ids are read before
 *     that kernel has completed and must not be written by it (nor by an
 *     earlier kernel still running because that one let it start early);
 *     q_rot and the cache are read after.  VH_FLAG_PLANNED: take the work list from the
 *     plan vh_decode_plan (with VH_FLAG_PLAN_THREE_CALL) wrote into this
 *     workspace for the same lengths, flags, page table, shape and num_ctas
 *     (see vh_decode_plan).
 * Softmax in fp32 with a running max, exp2 with log2(e) folded into the
 * scale; keys beyond seq_len (tail of the last page) are never used.  With
 * fp16, q_rot is split into an fp16 high part and residual for the tensor
 * cores, so its elements must lie within the fp16 range (|x| <= 65504).
 * Errors: VH_EINVAL (also for unknown flags), VH_EALIGN, VH_EWORKSPACE, VH_ECUDA. */
int vh_paged_decode_attn(const float* q_rot, const vh_e16* k_cache, const vh_e16* v_cache,
                         int64_t page_stride, int64_t token_stride, int64_t head_stride, int num_pages,
                         const int32_t* page_table, int max_pages_per_seq,
                         const int32_t* seq_lens, const int32_t* active,
                         vh_e16* out, float sm_scale, int num_ctas,
                         void* workspace, size_t workspace_bytes, int32_t* err_flag, unsigned flags,
                         int B, int Hq, int Hkv, int D, int page_size, void* stream);

/* Merge the partial results of split rows into out (e16 [B][Hq][D]; flags 0 or
 * VH_FLAG_FP16, as given to vh_paged_decode_attn).  Source: the same Fish
 * Speech section ("split-partial-combine" for long sequences, merged by the
 * online-softmax recurrence):
 * M = max_s lse_s, w_s = 2^(lse_s - M), o = sum_s w_s o_s / sum_s w_s (lse in
 * base 2).  Rows that were not split are left as vh_paged_decode_attn wrote
 * them.  Must run after vh_paged_decode_attn on the same stream with the same
 * workspace and the same shape / num_ctas arguments.
 * Errors: VH_EINVAL (also for unknown flags), VH_EALIGN, VH_EWORKSPACE, VH_ECUDA. */
int vh_decode_combine(const void* workspace, size_t workspace_bytes, vh_e16* out, int num_ctas,
                      unsigned flags, int B, int Hq, int Hkv, int D, int page_size, void* stream);

/* The whole decode step of one layer in ONE launch (the steps of
 * vh_rope_kv_append, vh_paged_decode_attn and vh_decode_combine, with their
 * sources; the pages run them as separate kernels): optional per-head RMSNorm
 * and RoPE of q and of the new key, append of the new key/value into the
 * cache, attention and the merge of split rows.  Same inputs and outputs as vh_rope_kv_append +
 * vh_paged_decode_attn + vh_decode_combine (apart from q_rot, which is not
 * written), with these differences:
 *   - the workspace must be zero-filled before its first use with this call
 *     (for example cudaMemsetAsync(workspace, 0, workspace_bytes)); it holds
 *     per-row counters that every completed call returns to zero, so later
 *     calls need no refill.  Refill it after a call that set VH_ERR_TIMEOUT;
 *   - a row whose position (positions[b], or seq_len-1) falls outside
 *     [0, max_pos) is treated like a padding row (zero output, no append) and
 *     VH_ERR_POS is set;
 *   - the new token's key is rotated and used by the CTA that owns the row's
 *     last tile, which also writes it (and v) to the cache slot; no other CTA
 *     reads that slot, so there is no ordering hazard inside the launch;
 *   - flags: VH_FLAG_FP16 and VH_FLAG_ROPE_INTERLEAVED as for
 *     vh_rope_kv_append, and VH_FLAG_PDL to launch as a programmatic
 *     dependent of the previous kernel on the stream, so that this launch's start-up (reading
 *     seq_lens, active, positions and page_table, planning the split)
 *     overlaps the end of that kernel.  Only valid when no kernel that may
 *     still run when this launch starts writes seq_lens, active, positions
 *     or page_table: the kernel launched immediately before on the same
 *     stream and, if that one is itself a programmatic dependent that lets
 *     its dependents start early (as this library's attention kernels do),
 *     the kernels before it, back to the last ordinary launch or copy (host
 *     copies in between are fine); everything else is read and written only
 *     after that kernel has completed.  The kernel itself always lets a
 *     following dependent launch start early.
 *     VH_FLAG_PDL_KV implies VH_FLAG_PDL and also requests the first tiles
 *     of the cached keys and values before that kernel has completed: valid
 *     only when it writes none of the cache pages this call reads (for
 *     instance the projection kernel of this layer, or this call for another
 *     layer's cache); the new token's slot is rewritten from k_new / v_new
 *     after the wait.  VH_FLAG_PLANNED: take the work list (tile ranges,
 *     row arrays, first page ids) from the plan vh_decode_plan wrote into
 *     this workspace, instead of deriving it from the lengths;
 *   - the workspace also holds that per-step plan: vh_decode_plan writes a
 *     region of it that this call only reads (and only with VH_FLAG_PLANNED);
 *   - VH_FLAG_HOST_IO (the pages have no counterpart: their runtime stages
 *     the step's inputs in device buffers): q, k_new, v_new, positions, seq_lens, active,
 *     page_table and out may be pinned host memory that the device reaches
 *     directly (on GB300, over the NVLink-C2C link to the Grace CPU): the
 *     kernel reads the step's inputs and writes its output in place, so a
 *     serving loop needs no separate host<->device copies and no copy-to-kernel
 *     dependencies in its graphs.  q rows are then loaded with plain loads
 *     (the other inputs always are), and with VH_FLAG_PDL the first q rows
 *     of each CTA are read before the wait on the previous kernel, like the
 *     lengths, flags and page ids: that kernel must not write q (inputs the
 *     host writes before the launch never are); cos_sin, the caches, the
 *     norm weights, err_flag and the workspace stay in device memory.  The caller keeps
 *     the host buffers unchanged until the launch has completed (double
 *     buffering across steps), as for any asynchronous read.
 * Errors: VH_EINVAL (also for unknown flags), VH_EALIGN, VH_EWORKSPACE,
 * VH_ENODEV, VH_ECUDA. */
int vh_decode_fused(const vh_e16* q, const vh_e16* k_new, const vh_e16* v_new,
                    const float* cos_sin, int max_pos, const int32_t* positions,
                    const float* q_norm_w, const float* k_norm_w, float norm_eps,
                    vh_e16* k_cache, vh_e16* v_cache, int64_t page_stride, int64_t token_stride,
                    int64_t head_stride, int num_pages, const int32_t* page_table, int max_pages_per_seq,
                    const int32_t* seq_lens, const int32_t* active,
                    vh_e16* out, float sm_scale, int num_ctas,
                    void* workspace, size_t workspace_bytes, int32_t* err_flag, unsigned flags,
                    int B, int Hq, int Hkv, int D, int page_size, void* stream);

/* Per-step plan of the attention work list, shared by every attention launch
 * of one decode step (all layers of a model see the same lengths, flags,
 * positions and page table).  The source pages have no counterpart: their
 * kernel picks its split from a host-side upper bound; here the split is a
 * device-side tile list (see vh_paged_decode_attn), and this call derives it
 * once per step instead of once per launch.
 * Writes into `workspace` (the one later passed to vh_decode_fused, or with
 * VH_FLAG_PLAN_THREE_CALL to vh_paged_decode_attn, with VH_FLAG_PLANNED): the
 * prefix sums of every row's 16-token tile count, the lengths and positions,
 * each CTA's tile range and the page ids of its first 64 tiles.  Rows that
 * take part: active rows with 1 <= seq_len <= max_pages_per_seq*P (others
 * flag VH_ERR_SEQLEN), and, for vh_decode_fused, a position (positions[b], or
 * seq_len-1) within [0, max_pos) (others flag VH_ERR_POS and are treated as
 * padding, as vh_decode_fused does).  max_pos is ignored with
 * VH_FLAG_PLAN_THREE_CALL.
 * Ordering: this kernel is an ordinary launch (it waits for all earlier work
 * on the stream) that lets no later kernel start before all of its CTAs
 * have exited, and each of its threads makes its plan writes visible at GPU
 * scope (a fence) before exiting, so every later launch on the stream,
 * programmatic dependents included, may read the plan before its own
 * dependency wait.  Call it again whenever
 * seq_lens, active, positions or page_table change (normally once per decode
 * step, after they are written and before the step's first attention
 * launch); a planned launch whose shape, num_ctas or path does not match the
 * plan's header ignores the plan and derives the work list itself, but one
 * made with stale lengths or page ids reads and appends where the old plan
 * says.  num_ctas: the value the attention launches get (0: automatic).
 * flags: VH_FLAG_FP16 (the element type of those launches) and
 * VH_FLAG_PLAN_THREE_CALL.
 * Errors: VH_EINVAL (also for unknown flags), VH_EALIGN, VH_EWORKSPACE,
 * VH_ENODEV, VH_ECUDA. */
int vh_decode_plan(const int32_t* positions, int max_pos, int num_pages, const int32_t* page_table,
                   int max_pages_per_seq, const int32_t* seq_lens, const int32_t* active, int num_ctas,
                   void* workspace, size_t workspace_bytes, int32_t* err_flag, unsigned flags,
                   int B, int Hq, int Hkv, int D, int page_size, void* stream);

/* Attention plus combine for callers that cannot allocate device memory.
 * The source pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory for a workspace (a runtime that only
 * hands out preallocated arenas, a plug-in inside a host process that owns
 * the CUDA context, a measurement that must not change the memory footprint).
 * Same arguments and result as vh_paged_decode_attn followed by
 * vh_decode_combine with flags 0 (bf16 cache and output) and token-major
 * pages (head_stride = D, so it takes no head_stride); page_table may be NULL
 * (a contiguous cache, as for the other calls).  There is no workspace: the
 * split-K partial
 * results go into one fixed array of VH_STATIC_SCRATCH_BYTES (8 MiB) compiled
 * into the library, which every GPU that loads the library keeps until the
 * process exits.  The call itself allocates and frees nothing.
 *   - The first call on each device looks up that device's address of the
 *     array (with that device current); make that first call before any
 *     stream capture.  A failed lookup is not remembered: the call returns
 *     VH_ECUDA and the next call looks again.
 *   - All calls share the one array and it keeps whatever the last call left
 *     there; nothing in it needs to start at zero.  Calls whose kernels can
 *     overlap on the GPU (different streams, or different host threads) race
 *     on the array and must be serialised by the caller.
 *   - A shape whose scratch need (vh_decode_workspace_bytes) exceeds
 *     VH_STATIC_SCRATCH_BYTES is rejected with VH_ESCRATCH before any launch.
 * Errors: VH_EINVAL, VH_EALIGN, VH_ESCRATCH, VH_ENODEV, VH_ECUDA. */
#define VH_STATIC_SCRATCH_BYTES (8u << 20)
int vh_paged_decode_attn_noalloc(const float* q_rot, const vh_bf16* k_cache, const vh_bf16* v_cache,
                                 int64_t page_stride, int64_t token_stride, int num_pages,
                                 const int32_t* page_table, int max_pages_per_seq,
                                 const int32_t* seq_lens, const int32_t* active,
                                 vh_bf16* out, float sm_scale, int num_ctas, int32_t* err_flag,
                                 int B, int Hq, int Hkv, int D, int page_size, void* stream);

/* Self-test of the failure path of the kernels' pipeline waits.  The source
 * pages have no counterpart: every wait of the attention kernels on an
 * mbarrier (a stage landing, a stage released, a partial result written) is
 * bounded by about a second of SM clock; when it runs out, the kernel ORs
 * VH_ERR_TIMEOUT into *err_flag and winds down instead of hanging the GPU.
 * This call launches one warp that runs that same bounded wait on a barrier
 * nothing ever arrives on, so the wait gives up (after about a second) and
 * VH_ERR_TIMEOUT is set; the CUDA context stays usable afterwards.
 * err_flag: device int32*, required (4-byte aligned).
 * Errors: VH_EINVAL (NULL err_flag), VH_EALIGN, VH_ENODEV, VH_ECUDA. */
int vh_selftest_wait_timeout(int32_t* err_flag, void* stream);

/* Static text for a return code (a host helper; the pages have no counterpart). */
const char* vh_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* VH_H */
