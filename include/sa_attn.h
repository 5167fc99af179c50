/*
 * sa_attn.h -- C ABI of the GB300 (sm_103a) RoPE + attention core of the
 * Stable Audio 3 DiT and SAME autoencoder.
 *
 * What one call computes, per (batch b, head h, query row i):
 *
 *   RoPE on q and k, rotate-half over the full head dim, in FP32, then cast
 *   back to the storage dtype (HF discussion #3 "fp16mixed attention-core fix",
 *   section "The bug": apply_rotary_pos_emb computes in FP32 and finishes
 *   with a cast to the output dtype; section "The fix": the rotation is
 *   multiplied out in FP32, then q and k are cast to fp16):
 *       theta_{p,i} = p * rope_base^(-2i/d),  i < d/2
 *       x'_i       = x_i cos(theta) - x_{i+d/2} sin(theta)
 *       x'_{i+d/2} = x_{i+d/2} cos(theta) + x_i sin(theta)
 *   then fused scaled-dot-product attention, non-causal, scale 1/sqrt(d), the
 *   softmax accumulated in FP32 (same page, "The bug": TensorRT's FMHA
 *   accumulates softmax in FP32):
 *       out_i = sum_j softmax_j(q'_i . k'_j / sqrt(d)) v_j
 *   Differential attention (lambda != NULL; HF discussion #6 "sm_120 SAME-L",
 *   section "How the kernels differ": two softmax maps sharing V, the
 *   subtraction kept in FP32 on FP32 accumulators):
 *       out_i = o(Q1,K1)_i - lambda_h * o(Q2,K2)_i
 *   Sliding window (window >= 0; the SAME-L diff_attn_swa window of the same
 *   page's "Three gotchas" is symmetric): key j is used for query i iff
 *   |i - j| <= window.  window < 0, or window >= L-1, is full attention.
 *
 * Conventions shared by every entry point:
 *   - Every function returns an sa_status; SA_OK is 0.  On any other status
 *     sa_last_error() returns a thread-local message that says what was wrong.
 *   - Device pointers must be CUDA device memory of the handle's device; all
 *     tensors are dense, C-contiguous, and 16-byte aligned.
 *   - Nothing is allocated and nothing is copied host<->device inside
 *     sa_rope_attn: it only encodes kernel arguments and enqueues two kernels
 *     on `stream`, so it can be captured into a CUDA graph.  When a host-side
 *     check fails, nothing is enqueued and `out` is not written.
 */
#ifndef SA_ATTN_H
#define SA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SA_API __attribute__((visibility("default")))
#else
#define SA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle: per-device state (FP32 RoPE frequency table, kernel
 * attributes, a 4-byte device error word).  Owned by the caller, freed by
 * sa_attn_destroy. */
typedef struct sa_attn_s* sa_attn_t;

/* The same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* sa_stream_t;

/* Element type of q, k, v and out.  SA_FP32 is the FP32-input form of SAME-L's
 * differential sliding-window attention (HF discussion #6 "sm_120 SAME-L",
 * "How the kernels differ": FP32 attention projections, both attention products
 * as TF32 MMAs with FP32 accumulation); it is accepted by sa_rope_attn,
 * sa_rope_attn_noalloc, sa_rope_qk and sa_attn_fwd for differential attention
 * (lambda != NULL, two maps) and refused with SA_ERR_UNSUPPORTED elsewhere. */
typedef enum { SA_FP16 = 0, SA_BF16 = 1, SA_FP32 = 2 } sa_dtype;

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size, bad value */
    SA_ERR_UNSUPPORTED = 2,     /* head dim other than 64, too many heads, wrong GPU */
    SA_ERR_CUDA = 3,            /* a CUDA runtime call or a launch failed */
    SA_ERR_DEVICE_TIMEOUT = 4,  /* a kernel gave up on a pipeline wait (see sa_attn_check) */
    SA_ERR_NO_DEVICE = 5,       /* no CUDA device, or the device index is out of range */
    SA_ERR_WORKSPACE = 6        /* workspace missing or smaller than sa_rope_attn_workspace_size */
} sa_status;

/* Largest H accepted by the differential path (lambda is passed by value). */
#define SA_MAX_DIFF_HEADS 128

/*
 * Create a handle on CUDA device `device`.  rope_base is the RoPE base
 * (10000 for Stable Audio 3); the FP32 frequency table rope_base^(-2i/64) is
 * computed here in double and rounded once.  The handle also holds the FP32
 * (cos, sin) table of positions 0..16383 (4 MiB of device memory, written here
 * once with the RoPE pass's arithmetic; skipped if it cannot be allocated),
 * which sa_rope_attn reads for small grids (below).  Fails with
 * SA_ERR_NO_DEVICE when there is no such device and SA_ERR_UNSUPPORTED when it
 * is not an sm_103 (GB300) part.  Restores the caller's current device before
 * returning.
 */
SA_API sa_status sa_attn_create(sa_attn_t* handle, int device, float rope_base);

/* Free the handle.  NULL is accepted.  Synchronizes the handle's device. */
SA_API sa_status sa_attn_destroy(sa_attn_t handle);

/*
 * Bytes of device workspace sa_rope_attn needs for this shape: the FP32
 * (cos, sin) table of sa_rope_table_bytes(L), the rotated and cast-back k
 * (B*H*nmaps*L*d elements of 2 bytes), each rounded up to 256 bytes, followed
 * by the split region of sa_attn_fwd_workspace_size bytes.  differential != 0
 * selects nmaps = 2.  Returns 0 for invalid sizes.
 */
SA_API size_t sa_rope_attn_workspace_size(int B, int H, int L, int d, int differential);

/*
 * Bytes of device workspace sa_rope_attn needs for this shape and element type.
 * SA_FP16 / SA_BF16: sa_rope_attn_workspace_size.  SA_FP32 (differential only):
 * the rotated q' and k' (B*H*2*L*d values of 4 bytes each), then v^T, the
 * transposed v ([B*H][2d][L4] FP32 values, L4 = L rounded up to a multiple of
 * 4), each rounded up to 256 bytes.  Returns 0 for invalid sizes or an
 * unsupported combination.
 */
SA_API size_t sa_rope_attn_workspace_bytes(int B, int H, int L, int d, int differential, sa_dtype dtype);

/*
 * Bytes of device workspace sa_attn_fwd needs for this element type:
 * sa_attn_fwd_workspace_size (optional) for SA_FP16 / SA_BF16; for SA_FP32 the
 * v^T region of sa_rope_attn_workspace_bytes (required).  0 for invalid sizes.
 */
SA_API size_t sa_attn_fwd_workspace_bytes(int B, int H, int L, int d, int differential, sa_dtype dtype);

/*
 * Bytes of the split region that sa_attn_fwd may be given: one 8-byte counter
 * per query block (256 rows standard, 128 differential) of every (batch,
 * head), rounded up to 256 bytes, then 160 FP32 partial-result slots of
 * 2*128*(d_v + 2) values.
 *
 * The attention kernel runs one CTA per query block.  When those leave the
 * GPU's last wave partly empty and the split region is given, each block of
 * that last wave is cut into k pieces of its key range (k as large as the wave
 * allows), one CTA each; the pieces leave FP32 partial results in the region
 * and the piece that finishes last merges them in a fixed order (results are
 * reproducible run to run).  The counters carry a per-launch tag and are
 * cleared by the launch that used them, so the region never needs clearing by
 * the caller (also across CUDA-graph replays).  Returns 0 for invalid sizes.
 */
SA_API size_t sa_attn_fwd_workspace_size(int B, int H, int L, int d, int differential);

/*
 * Enqueue RoPE + attention on `stream`: a pass rotates k into the workspace,
 * and the attention kernel rotates q as each Q tile arrives.  Usually the pass
 * also writes the (cos, sin) table the kernel reads.  When the attention grid
 * leaves SMs idle (fewer query blocks than SMs) and positions is NULL, the pass
 * runs on those SMs only and the kernel reads the handle's table, so its CTAs
 * start at once.  Either form gives the bits of sa_rope_qk followed by
 * sa_attn_fwd.
 *
 *   q, k      device, dtype.  Standard (lambda == NULL): [B, H, L, d].
 *             Differential (lambda != NULL): [B, H, 2, L, d]; map 0 is
 *             (Q1, K1), map 1 is (Q2, K2).
 *   v         device, dtype.  Standard: [B, H, L, d].  Differential:
 *             [B, H, L, 2d] (d_v = 128).
 *   positions device int32 [L] (shared by all batches and heads), or NULL for
 *             0..L-1.  Each is converted to FP32 before the angle product, which
 *             is exact for |p| < 2^24.
 *   out       device, dtype, [B, H, L, d_v].  Must not overlap any input.
 *   B, H, L   >= 1, L < 2^24, with B*H*L*d_v < 2^40.  d must be 64.
 *   window    < 0: full attention; >= 0: |i - j| <= window.
 *   lambda    host float[H] (H <= SA_MAX_DIFF_HEADS) or NULL.  Read during the
 *             call only (copied into the kernel arguments).
 *   dtype     SA_FP16 or SA_BF16 for q, k, v and out alike; or SA_FP32 for
 *             differential attention with FP32 q, k, v and out.  The FP32 form
 *             rotates q and k in FP32 in one pass that also transposes v (q', k',
 *             v^T in the workspace, each value rounded to TF32 to nearest, ties
 *             away from zero), then runs both attention products as kind::tf32
 *             MMAs (FP32 accumulate), the softmax and the lambda subtraction in
 *             FP32, and writes FP32 out.
 *   workspace device scratch of at least sa_rope_attn_workspace_bytes (for
 *             dtype) bytes, 16-byte aligned; contents on entry are ignored.
 *             Calls that use the same workspace must be ordered on the GPU
 *             (same stream).
 *   stream    CUDA stream; the call is asynchronous with respect to the host.
 *
 * Errors: SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_WORKSPACE from host
 * checks (nothing enqueued); SA_ERR_CUDA when a launch is rejected.  Device
 * side pipeline timeouts are reported later by sa_attn_check.
 */
SA_API sa_status sa_rope_attn(sa_attn_t handle,
                       const void* q, const void* k, const void* v,
                       const int32_t* positions,
                       void* out,
                       int B, int H, int L, int d,
                       int window,
                       const float* lambda,
                       sa_dtype dtype,
                       void* workspace, size_t workspace_bytes,
                       sa_stream_t stream);

/*
 * sa_rope_attn on HOST buffers: q, k, v are copied to the device, the path runs, and out is
 * copied back, all enqueued without blocking the host.  The (batch, head) planes are cut into
 * chunks of about 16 MiB of copies (two from 8 MiB up), at most 4 (more when a chunk would
 * exceed SA_MAX_DIFF_HEADS planes).  With one chunk everything runs on `stream` in order.  Otherwise
 * chunk c is copied in on the handle's copy-in stream, computed on compute stream c mod 4
 * (chunks on different streams run side by side on the GPU) and copied out on the copy-out
 * stream, so copies overlap computation.  Work enqueued on `stream` before the call is
 * ordered before it, and work enqueued on `stream` after it waits for the last output copy.
 *
 *   q, k, v, out  HOST memory, layouts as in sa_rope_attn.  Page-locked memory lets the
 *                 copies run asynchronously and overlap; pageable memory works but the
 *                 copies then serialise with the host.  out must stay valid (and unread)
 *                 until `stream` reaches the point after the call.
 *   positions     DEVICE int32 [L] or NULL, as in sa_rope_attn.
 *   workspace     DEVICE scratch, 16-byte aligned, of at least
 *                 sa_rope_attn_host_workspace_size bytes: device copies of q, k, v and out,
 *                 then one sa_rope_attn workspace per compute stream.
 *
 * The results have the bits of sa_rope_attn run on each chunk's planes (a chunk is a
 * contiguous range of the B*H planes, launched as B = 1 with its heads' lambdas).  Calls
 * that share a handle share its internal streams and are ordered on them.  Errors as
 * sa_rope_attn; SA_ERR_CUDA also when the handle's streams could not be created.
 */
SA_API size_t sa_rope_attn_host_workspace_size(int B, int H, int L, int d, int differential);

SA_API sa_status sa_rope_attn_host(sa_attn_t handle,
                                   const void* q, const void* k, const void* v,
                                   const int32_t* positions,
                                   void* out,
                                   int B, int H, int L, int d,
                                   int window,
                                   const float* lambda,
                                   sa_dtype dtype,
                                   void* workspace, size_t workspace_bytes,
                                   sa_stream_t stream);

/*
 * sa_rope_attn with a QK-RMSNorm in front of RoPE.  The pages run RMSNorm and
 * RoPE next to attention in FP32, so that variances cannot overflow fp16
 * (sa3_trt README, "Notes on the design"; the encoder/decoder tiers page,
 * "Where the quantization goes, per tier").  Here every row x of q and k (d
 * values, each map of the differential form alike) becomes, in FP32,
 *
 *   x_c * gamma_c / sqrt(mean_c(x_c^2) + eps),
 *
 * is then rotated as in sa_rope_attn and cast once to dtype; attention follows
 * unchanged.  The sum of squares is FP32, which holds every fp16 row; bf16
 * rows with a value of magnitude >= 2^63 overflow it (result undefined).
 *
 *   gamma_q, gamma_k  host float[d] (NULL: all ones), finite.  Read during the
 *                     call only (copied into the kernel arguments).
 *   eps               finite, >= 0.
 *
 * Everything else (arguments, workspace, errors) as sa_rope_attn; a bad gamma
 * or eps is SA_ERR_INVALID_ARG with nothing enqueued.
 */
SA_API sa_status sa_rope_attn_qknorm(sa_attn_t handle,
                                     const void* q, const void* k, const void* v,
                                     const int32_t* positions,
                                     const float* gamma_q, const float* gamma_k, float eps,
                                     void* out,
                                     int B, int H, int L, int d,
                                     int window,
                                     const float* lambda,
                                     sa_dtype dtype,
                                     void* workspace, size_t workspace_bytes,
                                     sa_stream_t stream);

/*
 * The two stages sa_rope_attn is made of, for callers that want them apart
 * (for instance to time the attention kernel alone, or to feed q/k that are
 * already rotated).  Same conventions, layouts and errors as sa_rope_attn.
 *
 * sa_rope_qk: q_rot = cast(RoPE_fp32(q)), k_rot = cast(RoPE_fp32(k)) for all
 *   B*H*nmaps planes of L rows (nmaps = 1 standard, 2 differential); q_rot and
 *   k_rot have the layout of q and k and must not overlap them.  With SA_FP32
 *   (nmaps = 2 only) the cast is the rounding to TF32 of sa_rope_attn's FP32
 *   form and q_rot, k_rot hold FP32 values.
 */
SA_API sa_status sa_rope_qk(sa_attn_t handle,
                            const void* q, const void* k,
                            const int32_t* positions,
                            void* q_rot, void* k_rot,
                            int B, int H, int L, int d, int nmaps,
                            sa_dtype dtype, sa_stream_t stream);

/*
 * sa_qknorm_rope_qk: sa_rope_qk with the QK-RMSNorm of sa_rope_attn_qknorm in
 *   front of the rotation (same gamma_q, gamma_k, eps rules).  Its q_rot, k_rot
 *   have the bits the normalised, rotated q and k have inside
 *   sa_rope_attn_qknorm.
 */
SA_API sa_status sa_qknorm_rope_qk(sa_attn_t handle,
                                   const void* q, const void* k,
                                   const int32_t* positions,
                                   const float* gamma_q, const float* gamma_k, float eps,
                                   void* q_rot, void* k_rot,
                                   int B, int H, int L, int d, int nmaps,
                                   sa_dtype dtype, sa_stream_t stream);

/*
 * The two stages as sa_rope_attn runs them: the pre-pass rotates k only and
 * the attention kernel rotates q in its prologue, as each Q tile arrives in
 * shared memory.
 *
 * sa_rope_table_bytes: bytes of cs_table, L * 32 (cos, sin) pairs of FP32
 *   (256 * L); 0 for invalid L.
 * sa_rope_k: k_rot = cast(RoPE_fp32(k)) (the layout of k) and the table of
 *   (cos, sin) of the FP32 angle fl(fl(p_l) * inv_freq[i]), i < 32,
 *   p_l = positions[l] or l, as float4 cs_table[m][l] = (cos_2m, cos_2m+1,
 *   sin_2m, sin_2m+1), m < 16 (rows of one pair-pair contiguous).
 *   cs_table: device, 16-byte aligned.
 * sa_attn_fwd_rope_q: attention (as sa_attn_fwd) on the raw q, rotated in the
 *   kernel's prologue with cs_table in the pre-pass's arithmetic, so the output
 *   has the same bits as sa_rope_qk followed by sa_attn_fwd; k_rot rotated
 *   already; workspace the optional split region of sa_attn_fwd.
 */
SA_API size_t sa_rope_table_bytes(int L);

SA_API sa_status sa_rope_k(sa_attn_t handle,
                           const void* k,
                           const int32_t* positions,
                           void* k_rot, void* cs_table,
                           int B, int H, int L, int d, int nmaps,
                           sa_dtype dtype, sa_stream_t stream);

SA_API sa_status sa_attn_fwd_rope_q(sa_attn_t handle,
                                    const void* q, const void* k_rot, const void* cs_table,
                                    const void* v, void* out,
                                    int B, int H, int L, int d,
                                    int window,
                                    const float* lambda,
                                    sa_dtype dtype,
                                    void* workspace, size_t workspace_bytes,
                                    sa_stream_t stream);

/*
 * sa_attn_fwd: scaled-dot-product attention (softmax in FP32; differential
 *   when lambda != NULL; sliding window when window >= 0) on q_rot, k_rot
 *   taken as already rotated.  workspace is optional: NULL runs one CTA per
 *   query block; otherwise it is a device split region (16-byte aligned) of at
 *   least sa_attn_fwd_workspace_size bytes (SA_ERR_WORKSPACE if smaller), and
 *   calls that use the same region must be ordered on the GPU (same stream).
 *   With SA_FP32 (lambda != NULL only) the attention stage of sa_rope_attn's
 *   FP32 form runs (TF32 products, one CTA per 128-row query block) after v
 *   is transposed into the workspace, which is then required: at least
 *   sa_attn_fwd_workspace_bytes bytes.
 */
SA_API sa_status sa_attn_fwd(sa_attn_t handle,
                             const void* q_rot, const void* k_rot, const void* v,
                             void* out,
                             int B, int H, int L, int d,
                             int window,
                             const float* lambda,
                             sa_dtype dtype,
                             void* workspace, size_t workspace_bytes,
                             sa_stream_t stream);

/*
 * The two stages of sa_rope_attn's FP32 form (SA_FP32, differential only), for
 * callers that want them apart.  Their composition has the bits of
 * sa_rope_attn.
 *
 * sa_rope_qkv_f32: q_rot, k_rot = RoPE of q, k ([B, H, 2, L, d] FP32) in FP32,
 *   rounded to TF32 (the layout of q and k); v_t = v ([B, H, L, 2d] FP32)
 *   transposed to [B*H][2d][L4] (L4 = L rounded up to a multiple of 4; keys
 *   L..L4-1 are zero), rounded to TF32.  All device, 16-byte aligned.
 * sa_attn_fwd_f32: the TF32 attention kernel on q_rot, k_rot and v_t as
 *   sa_rope_qkv_f32 leaves them; window and lambda as in sa_rope_attn.
 */
SA_API sa_status sa_rope_qkv_f32(sa_attn_t handle,
                                 const void* q, const void* k, const void* v,
                                 const int32_t* positions,
                                 void* q_rot, void* k_rot, void* v_t,
                                 int B, int H, int L, int d, sa_stream_t stream);

SA_API sa_status sa_attn_fwd_f32(sa_attn_t handle,
                                 const void* q_rot, const void* k_rot, const void* v_t,
                                 void* out,
                                 int B, int H, int L, int d,
                                 int window,
                                 const float* lambda,
                                 sa_stream_t stream);

/*
 * Size of the scratch array built into the library for sa_rope_attn_noalloc:
 * 64 MiB, enough for 2 * B*H*nmaps*L*64 two-byte elements up to that total
 * (every Stable Audio 3 shape here, up to B*H*nmaps*L = 262144 rows; a third
 * of that with SA_FP32, which also holds v^T).
 */
#define SA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * sa_rope_attn_noalloc: the same computation as sa_rope_attn, for callers
 * that cannot allocate device memory -- an engine plugin whose enqueue hook
 * only hands over tensor pointers and a stream, a real-time audio thread that
 * must not block in an allocator, a process whose device memory belongs to
 * another allocator.  The pages have no counterpart: this is an interface
 * convenience, not part of the method.
 *
 * It takes no workspace and allocates nothing: the rotated q', k' go to one
 * static device array of SA_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library keeps until the process exits.  A handle's
 * first call of this function looks up that array's device address (with the
 * handle's device current) and keeps it in the handle, so make that first call
 * before any stream capture.  All calls share the array: calls that may
 * overlap on the GPU race on it, so order them (one stream).  Nothing in it
 * needs clearing between calls.  The attention stage runs without the split
 * region of sa_rope_attn (one CTA per query block).
 *
 * Arguments, layouts and errors are those of sa_rope_attn, checked in the same
 * order.  Then a shape is accepted only if q' and k' fit the array:
 *   2 * round_up_256(B * H * maps * L * 64 * 2) <= SA_NOALLOC_SCRATCH_BYTES
 * (maps = 2 for differential attention, else 1), that is at most 262,144 rows
 * of 64 values (B * H * maps * L).  SA_FP32 also keeps v^T there:
 *   2 * round_up_256(B * H * 2 * L * 64 * 4)
 *     + round_up_256(B * H * 128 * round_up_4(L) * 4) <= SA_NOALLOC_SCRATCH_BYTES.
 * A larger shape is rejected with SA_ERR_WORKSPACE before anything is enqueued.
 */
SA_API sa_status sa_rope_attn_noalloc(sa_attn_t handle,
                                      const void* q, const void* k, const void* v,
                                      const int32_t* positions,
                                      void* out,
                                      int B, int H, int L, int d,
                                      int window,
                                      const float* lambda,
                                      sa_dtype dtype,
                                      sa_stream_t stream);

/*
 * Set the limit, in nanoseconds, of every pipeline wait inside the attention
 * kernel launched with this handle (default 1 s; at least 100 ns).  A wait
 * that runs out makes the kernel give up cleanly (it waits up to a second more
 * for its own copies and MMAs in flight, frees its tensor memory and exits) and
 * sets the error word that sa_attn_check reports as SA_ERR_DEVICE_TIMEOUT.
 * Meant for tests of that failure path; it changes no result when no wait
 * runs out.  Applies to launches enqueued after the call.
 */
SA_API sa_status sa_attn_set_timeout(sa_attn_t handle, unsigned long long timeout_ns);

/*
 * Synchronize the handle's device, then read and clear its device error
 * word.  SA_OK if no kernel since the last check gave up on a wait;
 * SA_ERR_DEVICE_TIMEOUT otherwise (its output is then unspecified).
 */
SA_API sa_status sa_attn_check(sa_attn_t handle);

/* Thread-local description of the last failure on this thread ("" if none). */
SA_API const char* sa_last_error(void);

/* Static name of a status code. */
SA_API const char* sa_status_string(sa_status status);

#ifdef __cplusplus
}
#endif

#endif /* SA_ATTN_H */
