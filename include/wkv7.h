/*
 * wkv7.h -- C ABI of the B300 (sm_103a) WKV7 state-recurrence library.
 *
 * The operation (per batch row b and head h, state S of D x D fp32 values,
 * row i = value index, column j = key index), for each token t in order:
 *
 *     sa_i  = sum_j S_ij a_j                    (state before the update)
 *     S_ij <- S_ij w_j + v_i k_j + sa_i b_j
 *     y_i   = sum_j S_ij r_j                    (state after the update)
 *
 * Source: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
 * architecture": the Forward listing (the update above, and a copy of the
 * state kept after every chunk of 32 tokens), the Backward listing (chunks
 * walked in reverse from those exact copies, the VJP giving dr, dw, dk, dv,
 * da, db, the previous state rebuilt as (h - v k - sa b) / w), and the note
 * that dividing by w amplifies rounding by (1/w)^N, which is why the copies
 * are kept every 32 tokens.  The listing leaves `sa` undefined; this library
 * reads it as the state times a, before the update.  The single-token decode
 * is the same update for T = 1 applied to a resident state ("RWKV-7 最新、最全
 * 的动态": the 7B model updates 32 x 64 heads of 64 x 64 state values per
 * token; "RWKV LM": an RNN continues from a passed state).
 *
 * Common conventions
 *   - Layouts are row-major and dense.  Per-token tensors are (B, T, H, D):
 *     element (b, t, h, j) at ((b*T + t)*H + h)*D + j.  States are (B, H, D, D):
 *     element (b, h, i, j) at ((b*H + h)*D + i)*D + j.  Checkpoints are
 *     (B, H, C, D, D) with C = wkv7_num_chunks(T, chunk).
 *   - r, w, k, v, a, b have dtype `in_dtype` (WKV7_F32 or WKV7_BF16).  All
 *     states, y and every gradient are fp32.  w is the decay multiplier, not its
 *     log, and must be > 0 where the backward divides by it.
 *   - Every pointer is a DEVICE pointer on the current CUDA device (memory the
 *     caller owns), 16-byte aligned.  The library calls no allocator and keeps
 *     no device memory of its own, with one exception: the fixed scratch array of
 *     wkv7_backward_noalloc (WKV7_NOALLOC_SCRATCH_BYTES, compiled into the
 *     library), which the CUDA runtime reserves on a device when the library's
 *     device code is loaded there (its first use on the device under the default
 *     lazy module loading) until the process exits.  Work is enqueued on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream) and is asynchronous: no
 *     call synchronises the device (except wkv7_debug_status).
 *   - D must be 64.  1 <= chunk <= 32.  B, H >= 1, T >= 0.
 *   - Outputs are fully overwritten (never accumulated into).  Outputs must not
 *     alias inputs or each other, except the in-place decode state.
 *   - Errors: every argument is checked on the host before anything is
 *     enqueued; a non-zero wkv7_status is returned and nothing runs.  A launch
 *     failure returns WKV7_ERR_CUDA (the CUDA error text is available from
 *     wkv7_last_cuda_error()).  Nothing aborts the process.
 */
#ifndef WKV7_H
#define WKV7_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { WKV7_F32 = 0, WKV7_BF16 = 1 } wkv7_dtype;

typedef enum {
    WKV7_OK = 0,
    WKV7_ERR_ARG = 1,      /* a required pointer is NULL, or a size is negative */
    WKV7_ERR_SHAPE = 2,    /* D != 64, chunk outside [1, 32], or sizes overflow the index range */
    WKV7_ERR_ALIGN = 3,    /* a pointer is not 16-byte aligned */
    WKV7_ERR_DTYPE = 4,    /* in_dtype is not WKV7_F32 / WKV7_BF16 */
    WKV7_ERR_CUDA = 5,     /* the CUDA runtime reported an error at launch */
    WKV7_ERR_TIMEOUT = 6,  /* a bounded device-side wait gave up (the workspace status word) */
    WKV7_ERR_WORKSPACE = 7, /* a workspace is smaller than its *_workspace_size */
    WKV7_ERR_SCRATCH_LIMIT = 8 /* wkv7_backward_noalloc: needs more than WKV7_NOALLOC_SCRATCH_BYTES */
} wkv7_status;

/* Number of checkpoints the forward writes: ceil(T / chunk); 0 for T == 0. */
int wkv7_num_chunks(int T, int chunk);

/*
 * Forward over T tokens.
 *   h0      (B,H,D,D) initial state, or NULL for zeros.
 *   y       (B,T,H,D) fp32 output, required.
 *   h_ckpt  (B,H,C,D,D) fp32 output or NULL (then no checkpoints are written --
 *           an inference prefill).  Entry c is the state after token
 *           min(T, (c+1)*chunk) - 1, so the last entry equals hT (T % chunk
 *           may be non-zero: the last chunk is then shorter).
 *   hT      (B,H,D,D) fp32 final state, or NULL.
 *   sa      (B,T,H,D) fp32 output or NULL: sa_t = S_{t-1} a_t for every token and
 *           state row (element (b,t,h,i) is row i).  Passing it to wkv7_backward
 *           selects the two-phase backward that reads it.
 *   workspace, workspace_bytes
 *           device scratch of at least wkv7_forward_workspace_size() bytes, 256-byte
 *           aligned, owned by the caller; or NULL / 0.  Used at chunk == 32 without sa
 *           (the chunk-operator forward): a parallel kernel forms every 32-token chunk's
 *           transition operator (S_end = S_start A_c + U_c, and the chunk's y from S_start)
 *           into it, 69632 bytes per (head, chunk) after a 256-byte header, with the
 *           chunk-internal part of y and the coupling matrices a later
 *           wkv7_backward_from_forward reuses; then one short chain per head applies them.  The
 *           header's first 4 bytes hold a status word: 0 after a call that completed
 *           normally; non-zero (WKV7_ERR_TIMEOUT) when a bounded wait inside the chain gave
 *           up (2 s), in which case the outputs are invalid.  Reading it is the caller's
 *           choice (it needs the stream synchronised).  Without a workspace at chunk 32 (no
 *           sa) the operators are formed inside the chain kernel, one chunk ahead (slower).
 *           With sa (or chunk != 32): 16-token sub-chunks when chunk % 16 == 0 and the B*H*2
 *           row blocks fit one wave of SMs, else token by token.
 * Results of every path agree with the token-by-token definition to ~1e-5 relative.
 * Source: Forward listing of "Metal kernel architecture" (see top of file).
 */
int wkv7_forward(int B, int T, int H, int D, int chunk, int in_dtype,
                 const void *r, const void *w, const void *k,
                 const void *v, const void *a, const void *b,
                 const float *h0, float *y, float *h_ckpt, float *hT, float *sa,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * The chunk-operator forward with y written in bf16 (round to nearest even) instead of fp32.
 *   y       (B,T,H,D) bf16 output (2 bytes per element), required when T > 0.
 *   workspace, workspace_bytes
 *           required (WKV7_ERR_ARG if NULL): as in wkv7_forward, and likewise usable by a
 *           following wkv7_backward_from_forward.
 *   chunk must be 32 (WKV7_ERR_SHAPE otherwise); there is no sa output.  Every other argument and
 *   result as wkv7_forward.  The state, the checkpoints and hT stay fp32; y is the fp32 value that
 *   wkv7_forward writes, rounded once to bf16 at the store (so it carries the bf16 rounding, a
 *   relative error up to 2^-9 per element, on top of the forward's ~1e-5).
 * Source: Forward listing of "Metal kernel architecture" (see top of file).
 */
int wkv7_forward_bf16_y(int B, int T, int H, int D, int chunk, int in_dtype,
                        const void *r, const void *w, const void *k,
                        const void *v, const void *a, const void *b,
                        const float *h0, void *y, float *h_ckpt, float *hT,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace wkv7_forward uses for these sizes (written to *bytes): 256 + 69632 per (head,
 * chunk) at chunk 32, 0 otherwise; returns a wkv7_status (the same size checks as wkv7_forward). */
int wkv7_forward_workspace_size(int B, int T, int H, int D, int chunk, size_t *bytes);

/*
 * The same forward, arguments and results as wkv7_forward (without a workspace), always
 * advanced token by token in fp32.  Kept callable for comparison and as the plain per-token path.
 */
int wkv7_forward_sequential(int B, int T, int H, int D, int chunk, int in_dtype,
                            const void *r, const void *w, const void *k,
                            const void *v, const void *a, const void *b,
                            const float *h0, float *y, float *h_ckpt, float *hT, float *sa,
                            void *stream);

/*
 * Checkpointed backward (vector-Jacobian product of wkv7_forward).
 *   h0      the forward's initial state, or NULL for zeros.
 *   h_ckpt  the forward's checkpoints (B,H,C,D,D), required when T > 0; the same
 *           chunk value must be passed.
 *   sa      the forward's `sa` output (B,T,H,D), or NULL: then each chunk is first
 *           run forward from its start checkpoint (h0 for the first) to recompute it.
 *   dy      (B,T,H,D) fp32 gradient of the loss w.r.t. y, required.
 *   dhT     (B,H,D,D) fp32 gradient w.r.t. hT, or NULL for zeros.
 *   dr, dw, dk, dv, da, db  (B,T,H,D) fp32 outputs, required.
 *   dh0     (B,H,D,D) fp32 gradient w.r.t. h0, or NULL (not written).
 *   workspace, workspace_bytes
 *           device scratch of at least wkv7_backward_workspace_size() bytes, 256-byte
 *           aligned, owned by the caller and reused freely between calls; or NULL / 0.
 *           With a workspace and no sa at chunk == 32 (the chunk-operator backward): a
 *           parallel kernel forms every chunk's transposed transition operator A_c^T and the
 *           chunk's dy contribution E_c into the workspace (the forward's layout); one short
 *           chain per head, last chunk to first, carries the state gradient G (w.r.t. the
 *           state after a chunk, from every later token) back through them, writing G at each
 *           chunk end over E_c, and dh0; then every chunk forms dr, dw, dk, dv, da, db at once
 *           in matrix form on tensor cores from the state before it (h_ckpt[c-1], or h0), G and
 *           the state after it, recomputing sa -- no state is divided by w.  Chunks whose
 *           decays are too strong for the matrix form (some w < 1/32, or a 32-token decay
 *           product below 1e-20) take the exact token-by-token passes.  Results ~1e-5 of
 *           exact.  The workspace header's status word is as in wkv7_forward.
 *           With a workspace and sa: the two-phase backward -- one pass over the sequence walks
 *           the state gradient (16 tokens per step in the closed form when chunk % 16 == 0 and
 *           the B*H*2 row blocks fit one wave of SMs, else token by token), then every chunk's
 *           column gradients at once by two token-by-token passes, with no division by w
 *           (~1e-7 of exact).
 *           Without a workspace a single pass does everything: each chunk is walked in reverse
 *           from the state at its end (the stored checkpoint with sa given; the chunk recomputed
 *           from its start checkpoint without), the earlier states rebuilt as
 *           (h - v k^T - sa b^T) / w (column j divided by w_j), which amplifies rounding by 1/w
 *           per token, as the page warns: ~5e-4 of exact at the workloads' decays (w >= 0.55),
 *           far worse where w is small (below ~0.05 it can exceed any useful tolerance); use a
 *           workspace there.
 * Sums are taken in a fixed order (no atomics): results are deterministic.
 * Source: Backward listing of "Metal kernel architecture" (see top of file).
 */
int wkv7_backward(int B, int T, int H, int D, int chunk, int in_dtype,
                  const void *r, const void *w, const void *k,
                  const void *v, const void *a, const void *b,
                  const float *h0, const float *h_ckpt, const float *sa,
                  const float *dy, const float *dhT,
                  float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                  float *dh0, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace wkv7_backward uses for these sizes (written to *bytes): at chunk 32 the larger of
 * the two-phase layout and the chunk-operator layout, else the two-phase one; returns a wkv7_status (the
 * same size checks as wkv7_backward). */
int wkv7_backward_workspace_size(int B, int T, int H, int D, int chunk, size_t *bytes);

/*
 * The chunk-operator backward that takes the transition operators from its forward instead of forming
 * them again (the forward's operators of a chunk are the backward's: A_c, and Q_c for E_c = DY^T Q_c^T),
 * and, with bf16 inputs, the coupling matrices M_ak, M_rb, M_rk and T = (I - M_ab)^-1 that the column
 * gradients use.
 *   fwd_workspace, fwd_workspace_bytes
 *           the workspace of the wkv7_forward call (chunk 32, no sa, with a workspace) that wrote
 *           h_ckpt from these same r..b and h0, untouched since; at least
 *           wkv7_forward_workspace_size() bytes, 256-byte aligned.  Required (WKV7_ERR_ARG if NULL).
 *           It is this call's only scratch and is consumed: E_c and G replace the forward's U_c and
 *           flags replace Q_c, so a second backward needs the forward run again.  A workspace that
 *           holds anything else gives meaningless gradients (nothing on the device can tell).
 *   Every other argument, layout and result as wkv7_backward with a workspace and no sa; chunk must
 *   be 32 (WKV7_ERR_SHAPE otherwise).  The walk reads A_c and Q_c from the forward's blocks and only
 *   E_c = DY^T Q_c^T is formed (by a first kernel, or, past 74 heads on 148 SMs, inside the walk itself)
 *   where wkv7_backward's first kernel forms A_c, Q_c and E_c; the column gradients skip forming the
 *   coupling matrices.  The walk sees the same
 *   A_c and E_c as wkv7_backward's on chunks in closed form (bit for bit); the matrices the forward
 *   formed differ from the column kernel's own in
 *   rounding only, so the gradients agree with wkv7_backward's to ~1e-6 relative.  The workspace
 *   header's status word is as in wkv7_forward.
 * Source: Backward listing of "Metal kernel architecture" (see top of file).
 */
int wkv7_backward_from_forward(int B, int T, int H, int D, int chunk, int in_dtype,
                               const void *r, const void *w, const void *k,
                               const void *v, const void *a, const void *b,
                               const float *h0, const float *h_ckpt,
                               const float *dy, const float *dhT,
                               float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                               float *dh0, void *fwd_workspace, size_t fwd_workspace_bytes, void *stream);

/* Bytes of device scratch the library owns for wkv7_backward_noalloc (128 MiB; see the conventions above). */
#define WKV7_NOALLOC_SCRATCH_BYTES (128u * 1024u * 1024u)

/*
 * The two-phase backward without any workspace argument and without allocating.
 *
 * For callers that cannot allocate device memory on the call path or hand the library
 * any: a host framework that gives an operator only its input and output buffers and no
 * allocator, or a latency-critical loop that must not risk cudaMalloc (which may
 * synchronise the device).  The scratch lives in one fixed array of
 * WKV7_NOALLOC_SCRATCH_BYTES inside the library, reserved on every GPU that loads the
 * library until the process exits.  There is no counterpart of this in the source pages:
 * it is a packaging of the same computation as wkv7_backward with a workspace.
 *
 *   Arguments, layouts and results: as wkv7_backward with a workspace, the same dispatch and
 *   bit-identical results; `sa` is required off 32-token chunks (there only the two-phase
 *   backward, which reads it, applies).  Problems whose wkv7_backward_workspace_size exceeds
 *   WKV7_NOALLOC_SCRATCH_BYTES return WKV7_ERR_SCRATCH_LIMIT (B12 T1024 H6 needs ~94 MB;
 *   use wkv7_backward with a workspace for larger ones).
 *   Each call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress), so a device reset between calls is harmless.  The first call on
 *   a device may load the library's device code there (lazy loading: that reserves the
 *   array); make it before capturing a stream on that device.
 *   All calls share the one array and it keeps the previous call's contents; nothing in
 *   it needs clearing (each call writes every scratch value before reading it).  Calls
 *   whose work overlaps on the GPU (different streams, or different host threads) race on
 *   the array: serialise them.
 */
int wkv7_backward_noalloc(int B, int T, int H, int D, int chunk, int in_dtype,
                          const void *r, const void *w, const void *k,
                          const void *v, const void *a, const void *b,
                          const float *h0, const float *h_ckpt, const float *sa,
                          const float *dy, const float *dhT,
                          float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                          float *dh0, void *stream);

/*
 * One decode token for B sequences of H heads, state updated in place.
 *   state   (B,H,D,D) fp32, read and overwritten; same layout as h0 / hT.
 *   r..b    (B,H,D) in in_dtype (the (B,T,H,D) layout with T = 1).
 *   y       (B,H,D) fp32 output, required.
 * Equal to wkv7_forward with T = 1, h0 = state, hT = state.
 */
int wkv7_decode(int B, int H, int D, int in_dtype, float *state,
                const void *r, const void *w, const void *k,
                const void *v, const void *a, const void *b,
                float *y, void *stream);

/* Static text for a wkv7_status value. */
/* ---- device-side index checks (no counterpart in the pages: a stand-in for a memory checker)
 * A library built with WKV7_DEBUG_CHECKS (build.py --debug: libwkv7_debug.so) checks the indices its
 * kernels derive (shared-memory operand rows and columns, global rows, tile and block indices) and,
 * instead of making an out-of-range access, records it in a status word of the kernel's source file and
 * skips the access (or reads a safe address); no kernel traps.
 *   wkv7_debug_status: synchronizes the device, then ORs and clears every file's word into *word: 0 = no
 *     failed check since the last call; bit 0 an operand helper, bit 1 the chunk-operator prep, bit 2 its
 *     chain, bit 3 the matrix column kernel, bit 4 its token-by-token companion, bit 5 other kernels.
 *     Release builds write 0.  WKV7_ERR_ARG for a NULL word; WKV7_ERR_CUDA if the device reports an error.
 *   wkv7_debug_enabled: 1 for a debug build, else 0. */
int wkv7_debug_status(unsigned *word);
int wkv7_debug_enabled(void);

const char *wkv7_strerror(int status);

/* Text of the last CUDA error seen by this library on the calling thread ("" if none). */
const char *wkv7_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int wkv7_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_H */
