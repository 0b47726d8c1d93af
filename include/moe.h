/*
 * moe.h -- C ABI of the GB300 (sm_103a) dropless, sorted-dispatch
 * mixture-of-experts layer: forward pass and train step (value and gradients
 * with respect to the input and every parameter).
 *
 * The layer (benchmark pages kernel_gmm_gpu.json / gpu_nn.json /
 * gpu_moe_h100.json; the parameter count on gpu_nn.json, results[suite=moe]
 * .params = 12,587,008 = E*3*d*h + d*E for E=8, d=512, h=1024, fixes the
 * structure):
 *
 *   logits = x W_r                               (route piece)
 *   idx[t, 0..k-1] = top-k experts of logits[t]  (ties -> lower expert index,
 *                    slots in descending logit order)
 *   gates[t, :]    = softmax(logits[t, idx[t, :]])
 *   pairs p = t*k + j sorted by expert, stable  (sort_permute piece)
 *   H_r = silu(x_t W_gate[e]) * (x_t W_up[e]),  O_r = H_r W_down[e]
 *                                               (experts_grouped_swiglu piece)
 *   y[t] = sum_j gates[t, j] O_{row(t, j)} + shared(x[t])
 *                                               (unpermute_combine piece; the
 *                    shared expert is the `shared` field of gpu_moe_h100.json)
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  Every
 *   tensor is dense and row-major.  Weights: w_router [d, E]; w_gate, w_up
 *   [E, d, h]; w_down [E, h, d]; ws_gate, ws_up [d, hs]; ws_down [hs, d].
 * - Activations, weights and their gradients move in 16-byte vectors and
 *   bulk copies: each of those arrays must start on a 16-byte boundary
 *   (MOE_ERR_INVALID_ARG otherwise).  Index, gate and logit arrays need only
 *   their element alignment.
 * - dtype MOE_F32: every activation, weight and gradient is float32.
 *   dtype MOE_BF16: x, y, dy, dx, weights and the saved activations are
 *   bfloat16; logits, gates and every weight gradient are float32.
 *   Accumulation is float32 in both.
 * - The library allocates nothing.  Scratch is the caller's workspace of
 *   moe_workspace_bytes() bytes (256-byte aligned).  The SAME workspace must
 *   be passed to every call of one layer invocation: moe_permute writes the
 *   dispatch tables (expert-padded row map, tile list) into it and the later
 *   calls read them; the forward leaves state there that moe_backward reads.
 * - Everything is enqueued on `stream`; no call synchronises the host except
 *   moe_read_device_status.
 * - Arguments are validated before anything is launched.  On a non-OK status
 *   nothing was launched and no output was written.
 * - Kernel-side failures (a bounded wait that ran out, a device-side index
 *   check) do not fault: they set a code in the workspace that
 *   moe_read_device_status returns.
 * - Expert-sorted activation buffers (h_buf, a_gate_saved, a_up_saved) hold
 *   moe_padded_rows() rows: each expert's rows start on a multiple of 256 and
 *   the rows between experts are padding.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad mode          */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape, dtype)  */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed         */
  MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out            */
  MOE_ERR_DEVICE_CHECK = 6   /* device: an index check failed             */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  MOE_FWD_ONLY = 0,      /* forward only: nothing saved for a backward     */
  MOE_SAVE_FOR_BWD = 1,  /* forward of a train step: pre-activations saved */
  MOE_SHARED_READY = 2   /* moe_combine flag (OR-ed into the mode): the
                            shared expert's output was already produced by
                            moe_shared_ffn_fwd on this workspace          */
} moe_mode;

typedef struct {
  int64_t tokens;        /* T >= 0                                      */
  int32_t d_model;       /* d, multiple of 64                            */
  int32_t d_hidden;      /* h, expert hidden width, multiple of 64       */
  int32_t experts;       /* E, 1..256                                    */
  int32_t top_k;         /* k, 1..min(E, 32)                             */
  int32_t shared_hidden; /* hs, 0 = no shared expert, else multiple of 64 */
  int32_t dtype;         /* moe_dtype                                    */
  int32_t capacity;      /* pairs an expert takes: 0 = dropless (every
                            pair); C > 0 = capacity routing: each expert
                            keeps its first C pairs in increasing pair id
                            p = t*k + j and drops the rest               */
} moe_dims;

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

/* Workspace bytes needed by every call of one layer invocation in `mode`
 * (MOE_SAVE_FOR_BWD also covers moe_backward).  *bytes is written on OK. */
moe_status moe_workspace_bytes(const moe_dims* dims, int mode, size_t* bytes);

/* Row capacity of the expert-sorted activation buffers:
 * T*k + E*127 rounded up to 128. */
moe_status moe_padded_rows(const moe_dims* dims, int64_t* rows);

/* Passage: the `route` piece of kernel_gmm_gpu.json (pieces suite) and the
 * `top_k` field of gpu_moe_h100.json; the bias-free d x E router from the
 * parameter count of gpu_nn.json.
 * Router: logits = x W_r (+ router_bias) (float32 accumulate), then per
 * token the top-k experts (ties to the lower index, descending slots) and
 * the softmax of the selected logits.
 *   x          [T, d]  (dtype)            w_router [d, E] (dtype)
 *   router_bias [E]    f32, nullable: a fixed per-expert offset added to the
 *              computed logits (it skews the routing; the layer trains no
 *              bias, so moe_backward returns no gradient for it); ignored
 *              with logits_in
 *   logits_in  [T, E]  f32, nullable: when given, the GEMM is skipped and
 *              the selection is made on these logits (fed-logits mode;
 *              x and w_router may then be NULL)
 *   logits_out [T, E]  f32, nullable: receives the logits used
 *   topk_idx   [T, k]  int32 out          gates [T, k] f32 out
 * Logits must be finite (a NaN makes the selection unspecified). */
moe_status moe_route(const moe_dims* dims, const void* x, const void* w_router,
                     const float* router_bias, const float* logits_in, float* logits_out,
                     int32_t* topk_idx, float* gates, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* Passage: the `sort_permute` piece and the `sorted` dispatch of
 * kernel_gmm_gpu.json.
 * Counting sort of the T*k pairs p = t*k + j by expert topk_idx[p],
 * stable in p.
 *   counts   [E]     int32 out: pairs per expert
 *   offsets  [E+1]   int32 out: exclusive prefix sum of counts
 *   perm     [T*k]   int32 out: perm[r] = pair at sorted position r
 *   inv_perm [T*k]   int32 out: inv_perm[perm[r]] = r
 * Also writes the expert-padded row map and the tile list into the
 * workspace for the grouped calls.  Entries of topk_idx must lie in
 * [0, E) and be distinct per token.  With dims->capacity = C > 0 only the
 * kept pairs (each expert's first C in increasing p) are sorted: counts and
 * offsets count kept pairs, perm[r] = -1 for r >= offsets[E] and
 * inv_perm[p] = -1 for a dropped pair.  A dropped pair adds nothing to y;
 * the gates stay the softmax over all k selected logits, so the router
 * gradient still reaches a dropped slot through its token's kept slots.
 * An out-of-range index is reported (MOE_ERR_DEVICE_CHECK) and its pair is
 * treated as dropped. */
moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Passage: the `experts_grouped_swiglu` piece of kernel_gmm_gpu.json (the
 * three bias-free 512 x 1024 matrices per expert of gpu_nn.json's count).
 * Grouped SwiGLU experts over the expert-sorted rows (the token rows are
 * first gathered into expert-sorted order inside the workspace):
 *   h_buf[r] = silu(x_t W_gate[e]) * (x_t W_up[e])     [padded_rows, h] (dtype)
 *   then, for the down projection, gates[t, j] * (h_buf[r] W_down[e]) is
 *   kept in the workspace as pair (t, j)'s share of y[t], for moe_combine.
 * In MOE_SAVE_FOR_BWD mode a_gate_saved / a_up_saved [padded_rows, h]
 * (dtype) receive x_t W_gate[e] and x_t W_up[e]; in MOE_FWD_ONLY they may
 * be NULL.  gates is moe_route's output. */
moe_status moe_grouped_ffn_fwd(const moe_dims* dims, int mode, const void* x,
                               const float* gates, const void* w_gate, const void* w_up,
                               const void* w_down, void* h_buf, void* a_gate_saved,
                               void* a_up_saved, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* Passage: the `unpermute_combine` piece of kernel_gmm_gpu.json; the shared
 * expert is the `shared: 1024` field of gpu_moe_h100.json; the value
 * sum(y * upstream) is the train step's value of the value_and_grad
 * description of gpu_moe_h100.json.
 * Combine: y[t] = shared(x_t) + sum over slots j of the pairs' shares left
 * by moe_grouped_ffn_fwd, summed in slot order and cast to dtype, where
 * shared(x) = (silu(x Ws_gate) * (x Ws_up)) Ws_down when hs > 0 (its
 * weights are ignored and may be NULL when hs == 0).
 *   y [T, d] (dtype) out
 *   hs_buf [T, hs] (dtype) scratch for the shared hidden activations
 *                          (NULL when hs == 0)
 *   as_gate_saved, as_up_saved [T, hs] (dtype): saved shared
 *                          pre-activations in MOE_SAVE_FOR_BWD, else NULL
 *   upstream [T, d] (dtype), nullable; when given, *loss (f32, device)
 *   receives sum(y * upstream), the train step's value, reduced in a fixed
 *   order.  The result is bit-identical from run to run.
 * With MOE_SHARED_READY OR-ed into `mode`, the shared expert's output is
 * taken from the workspace, where moe_shared_ffn_fwd left it (the caller
 * orders that call before this one); x, the shared weights and its buffers
 * are then ignored. */
moe_status moe_combine(const moe_dims* dims, int mode, const void* x, const void* ws_gate,
                       const void* ws_up, const void* ws_down, void* y, void* hs_buf,
                       void* as_gate_saved, void* as_up_saved, const void* upstream, float* loss,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Passage: the value_and_grad description of gpu_moe_h100.json (gradients
 * with respect to the input and every parameter).
 * Backward of the train step for L = sum(y * dy):
 *   inputs : dy [T, d], x, all weights, topk_idx, gates, and what a
 *            MOE_SAVE_FOR_BWD forward that used the same workspace left:
 *            its pre-activations a_gate_saved / a_up_saved [padded_rows, h]
 *            and h_saved [padded_rows, h] (the h_buf of moe_grouped_ffn_fwd),
 *            and for the shared expert as_gate_saved / as_up_saved and
 *            hs_saved [T, hs] (the hs_buf of moe_combine; all three NULL
 *            when hs == 0)
 *   outputs: dx [T, d] (dtype); dw_router [d, E], dw_gate/dw_up [E, d, h],
 *            dw_down [E, h, d], dws_gate/dws_up [d, hs], dws_down [hs, d]
 *            (all f32; the dws_* NULL when hs == 0).  Outputs are
 *            overwritten, not accumulated.
 * The router gradient follows from the softmax over the selected logits;
 * experts that were not selected get no logit gradient.  The saved
 * buffers are read only. */
moe_status moe_backward(const moe_dims* dims, const void* dy, const void* x,
                        const void* w_router, const void* w_gate, const void* w_up,
                        const void* w_down, const void* ws_gate, const void* ws_up,
                        const void* ws_down, const int32_t* topk_idx, const float* gates,
                        const void* a_gate_saved, const void* a_up_saved, const void* h_saved,
                        const void* as_gate_saved, const void* as_up_saved,
                        const void* hs_saved, void* dx, float* dw_router, float* dw_gate,
                        float* dw_up, float* dw_down, float* dws_gate, float* dws_up,
                        float* dws_down, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/* The shared expert on its own, so that it can run on another stream beside
 * the routed experts (the two share no buffer):
 *
 * moe_shared_ffn_fwd: the shared expert's forward (the `shared` field of
 * gpu_moe_h100.json): its output rows go to the workspace for a following
 * moe_combine(mode | MOE_SHARED_READY); hs_buf / as_gate_saved /
 * as_up_saved as in moe_combine.  Nothing to do (MOE_OK) when hs == 0.
 *
 * moe_shared_backward: the shared expert's share of the value_and_grad
 * backward (gpu_moe_h100.json): dws_gate / dws_up [d, hs], dws_down [hs, d]
 * (f32, overwritten) and its rows of dx, which it leaves in the workspace
 * for moe_backward_routed.  Reads what the forward on this workspace saved.
 *
 * moe_backward_routed: moe_backward without the shared expert: the routed
 * experts' and the router's gradients, and dx, which adds the shared
 * expert's rows when hs > 0.  shared_done (nullable) is an event recorded
 * after moe_shared_backward was enqueued (on any stream): the kernel that
 * forms dx waits for it; with NULL the caller orders the two calls itself
 * (e.g. both on one stream, the shared one first). */
moe_status moe_shared_ffn_fwd(const moe_dims* dims, int mode, const void* x, const void* ws_gate,
                              const void* ws_up, const void* ws_down, void* hs_buf,
                              void* as_gate_saved, void* as_up_saved, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);
moe_status moe_shared_backward(const moe_dims* dims, const void* dy, const void* x,
                               const void* ws_gate, const void* ws_up, const void* ws_down,
                               const void* as_gate_saved, const void* as_up_saved,
                               const void* hs_saved, float* dws_gate, float* dws_up,
                               float* dws_down, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);
moe_status moe_backward_routed(const moe_dims* dims, const void* dy, const void* x,
                               const void* w_router, const void* w_gate, const void* w_up,
                               const void* w_down, const int32_t* topk_idx, const float* gates,
                               const void* a_gate_saved, const void* a_up_saved,
                               const void* h_saved, void* dx, float* dw_router, float* dw_gate,
                               float* dw_up, float* dw_down, cudaEvent_t shared_done,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Caps the number of SMs that the persistent kernels launched afterwards
 * by the calling host thread may occupy (0: every SM).  With the shared
 * expert on a second stream, the two streams' kernels then run side by side
 * on disjoint shares of the GPU instead of one waiting for the other.  The
 * results do not depend on the cap (work schedules that fix a summation
 * order are sized for the whole device).  A launch recorded into a CUDA
 * graph keeps the cap it was recorded under.  Not a device setting: it
 * only sizes this thread's grids. */
moe_status moe_set_sm_limit(int sms);

/* Synchronises `stream`, then returns the device-side status recorded in
 * the workspace since the last moe_permute (MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE_CHECK) and clears it.  *detail (nullable) receives a
 * kernel-specific detail word. */
moe_status moe_read_device_status(void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream, int32_t* detail);

/* moe_permute_noalloc: the same counting sort as moe_permute (counts,
 * offsets, perm, inv_perm; identical results, also for rejected expert
 * indices) for callers that cannot
 * allocate device memory -- code running where cudaMalloc is unavailable or
 * not allowed, such as an engine plugin handed no workspace, a serving loop
 * whose memory was reserved up front by another allocator, or a caller that
 * must not risk the implicit device synchronisation of an allocation.  The
 * benchmark pages have no counterpart to this entry; it exists for them.
 *
 * It takes no workspace.  Its scratch is one array of 4 MiB + 1.5 KiB inside
 * the library (a __device__ variable: every GPU that loads the library keeps
 * it until the process exits).  It is sized for (T*k / 512, rounded up) x E
 * <= 524288, e.g. up to 2^20 pairs with 256 experts or 2^22 pairs with 64;
 * larger problems return MOE_ERR_UNSUPPORTED before anything is launched,
 * and so does capacity routing (dims->capacity != 0): it sorts every pair.
 * It does not write the expert-padded tables the grouped calls read, so it
 * is not a substitute for moe_permute inside a layer invocation.
 *
 * All calls share the array and each call leaves its contents behind;
 * calls that overlap on the GPU (other streams, unsynchronised threads)
 * race.  The first call on a device looks up the array's device address,
 * which loads the library's device code there; make that first call before
 * any stream capture.  An expert index outside [0, E) is treated as
 * moe_permute treats it: its pair gets no sorted position (inv_perm = -1)
 * and perm reads -1 past offsets[E]; this entry has no status word, so
 * those -1 entries are the only report. */
moe_status moe_permute_noalloc(const moe_dims* dims, const int32_t* topk_idx, int32_t* counts,
                               int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                               cudaStream_t stream);

/* Kernel timing records, a measurement aid outside the layer itself: while
 * enabled, every kernel the library launches is bracketed by two CUDA events
 * recorded on its stream.  Enabling or disabling discards earlier records.
 * Not thread-safe with respect to concurrent launches from several threads. */
moe_status moe_profile_enable(int enable);

/* Aggregates the records per kernel name (synchronising on them): up to
 * max_entries names of 64 bytes each (NUL-terminated) into `names`, launch
 * counts into `launches` and summed device milliseconds into `total_ms`
 * (each nullable); *n_entries receives the number of distinct kernels. */
moe_status moe_profile_read(int max_entries, char* names, int64_t* launches, double* total_ms,
                            int* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
