/*
 * gla.h — C ABI of libgla.so: Simple Gated Linear Attention (Simple GLA) on
 * NVIDIA GB300 (sm_103a).
 *
 * The method (page "线性注意力模型如何实现固定推理状态" — Beyond the KV cache:
 * training and serving i14's Laplace 3B linear attention model on AWS
 * Trainium2 — section "i14 与 Laplace 3B 架构", GLA mixer and decay scheme):
 * every head h keeps a dk x dv matrix state S and a fixed, non-learned scalar
 * decay lambda_h = exp(log_decay[h]) in (0, 1].  For each token t
 *
 *     S_t = lambda_h * S_{t-1} + k_t^T v_t          (state update)
 *     o_t = q_t S_t                                 (read-out, after the update)
 *
 * with k_t, q_t in R^{1 x dk}, v_t, o_t in R^{1 x dv}.  There is no extra
 * scale: any 1/sqrt(dk) belongs to the caller's q.
 *
 * Conventions shared by every entry point
 *   - Layouts are row-major with the innermost dimension last.
 *   - Every pointer argument is a DEVICE pointer of the current CUDA device and
 *     must be 16-byte aligned (GLA_ERR_ALIGN otherwise); gla_chunk_fwd_host
 *     alone takes host pointers, with no alignment rule.  The caller owns every
 *     buffer; the library never frees or keeps a caller pointer.
 *   - "bf16" means IEEE-754 binary16-bfloat (torch.bfloat16); "f32" float.
 *     States (h0, hT, state_inout) and log_decay are always f32, and all
 *     accumulation is f32.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: the return value covers host-side argument checks and the
 *     launch.  Failures found on the device (a bounded wait that ran out, a bad
 *     cu_seqlens entry) are recorded in a device status word that
 *     gla_last_device_status() returns and clears.
 *   - Inputs and outputs must not overlap, except state_inout, which is
 *     updated in place.
 *   - Thread-safe: the only global state is a per-device capability cache and
 *     the device status word.
 *   - The library needs an sm_103a device (GB300); on any other device every
 *     compute entry point returns GLA_ERR_UNSUPPORTED.
 */
#ifndef GLA_H_
#define GLA_H_

#include <stdint.h>

#if defined(__GNUC__)
#define GLA_API __attribute__((visibility("default")))
#else
#define GLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GLA_OK = 0,
    GLA_ERR_ARG = -1,          /* null pointer, non-positive size, inconsistent sizes */
    GLA_ERR_UNSUPPORTED = -2,  /* shape / chunk outside what the kernels handle, or not sm_103a */
    GLA_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned */
    GLA_ERR_LAUNCH = -4,       /* a CUDA call or kernel launch failed */
    GLA_ERR_TIMEOUT = -5,      /* device: a bounded pipeline wait gave up (reported by gla_last_device_status) */
    GLA_ERR_NOMEM = -6,        /* stream-ordered scratch allocation failed */
    GLA_ERR_DEVICE_ARG = -7,   /* device: cu_seqlens not non-decreasing / out of [0, T] (gla_last_device_status) */
    GLA_ERR_SCRATCH_LIMIT = -8 /* gla_chunk_fwd_noalloc: the problem needs more than its fixed scratch array */
} gla_status;

/* Output gate of the *_gated entry points (page "线性注意力模型如何实现固定推理状态", section
 * "i14 与 Laplace 3B 架构", QKVG projection: the projection also yields a gate g_t of H x dv values per
 * token, applied after the mixer; the page gives no formula, so both usual forms are offered). */
typedef enum {
    GLA_GATE_SILU = 0,    /* out = o * g / (1 + exp(-g))   (swish) */
    GLA_GATE_SIGMOID = 1  /* out = o / (1 + exp(-g)) */
} gla_gate_kind;

/*
 * gla_chunk_fwd — chunkwise-parallel prefill / training forward, bf16 q, k, v, out.
 *
 * Computes, for every sequence and head, the recurrence above over all tokens
 * in chunks of `chunk` tokens (page "线性注意力模型如何实现固定推理状态",
 * section "挑战 1", chunked GLA and Figure 3): within chunk c of length L
 * (local positions i, j)
 *     O_c = ((Q_c K_c^T) .* D) V_c + diag(lambda^(i+1)) Q_c S_{c-1},
 *           D_ij = lambda^(i-j) if j <= i else 0,
 *     S_c = lambda^L S_{c-1} + K_c^T diag(lambda^(L-1-j)) V_c,
 * which equals the token-by-token recurrence up to rounding.
 *
 * Arguments
 *   q, k       [B, T, H, dk] bf16           (packed: [1, T, H, dk])
 *   v          [B, T, H, dv] bf16           (packed: [1, T, H, dv])
 *   log_decay  [H] f32, natural log of lambda_h, each <= 0 and finite
 *   h0         [B, H, dk, dv] f32 initial state, or NULL for zeros
 *   out        [B, T, H, dv] bf16, written
 *   hT         [B, H, dk, dv] f32 final state, written; or NULL to skip
 *   B, T, H    batch, tokens per sequence, heads (all > 0)
 *   dk, dv     key / value head sizes: 16 <= dk <= 256 and 16 <= dv <= 512,
 *              both multiples of 8
 *   chunk      chunk length 16, 32, 64 or 128: 128 and 64 select the
 *              tensor-core kernel (tcgen05/TMEM, fed by TMA) when 32 | dk <= 128
 *              and 64 | dv <= 192 and its tiles fit in shared memory (every
 *              such shape but dk = 128 with dv = 192; chunk 64 as two chunks
 *              per 128-row tile, see gla_chunk_kernel); 16 and 32, and any
 *              chunk outside that envelope, run the SIMT kernel, which splits
 *              a chunk that does not fit in shared memory in halves.
 *              gla_chunk_kernel tells which kernel a call will run
 *   cu_seqlens NULL for a dense batch.  Otherwise a DEVICE int32 array [B+1]
 *              of packed sequence offsets: sequence s is rows
 *              cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed [1, T, ...]
 *              tensors, B is the number of sequences, T the total rows, and
 *              h0 / hT are [B, H, dk, dv].  Chunks restart at every sequence
 *              start; an empty sequence gets hT = h0.  Offsets must be
 *              non-decreasing within [0, T]; a sequence that violates this is
 *              skipped and GLA_ERR_DEVICE_ARG is recorded on the device.
 *   stream     cudaStream_t
 * Long dense sequences with few (sequence, head) chains may be split into
 * segments whose boundary states are found in a first pass; that schedule
 * takes stream-ordered scratch (cudaMallocAsync / cudaFreeAsync on `stream`,
 * GLA_ERR_NOMEM on failure).  Returns a gla_status.
 */
GLA_API int gla_chunk_fwd(const void *q, const void *k, const void *v, const float *log_decay,
                  const float *h0, void *out, float *hT, int B, int T, int H, int dk, int dv,
                  int chunk, const int32_t *cu_seqlens, void *stream);

/*
 * gla_chunk_fwd_gated — gla_chunk_fwd with the output gate fused into the write of out:
 *     out[t, h, :] = o_t,h * f(g[t, h, :])   elementwise, f per gate_kind (gla_gate_kind)
 * where o is what gla_chunk_fwd computes; hT is unchanged by the gate.
 *   g          [B, T, H, dv] bf16 (packed [1, T, H, dv]), the layout of out; device, 16-byte aligned;
 *              read only (it may not alias out)
 *   gate_kind  GLA_GATE_SILU or GLA_GATE_SIGMOID (else GLA_ERR_ARG)
 *   all other arguments, the schedules and the errors: as gla_chunk_fwd.
 * The gate costs one extra read of H * dv bf16 per token (1,536 instead of 1,152 bytes per token-head
 * at dk 96, dv 192) and no extra launch.  Returns a gla_status.
 */
GLA_API int gla_chunk_fwd_gated(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                                const float *log_decay, const float *h0, void *out, float *hT, int B, int T,
                                int H, int dk, int dv, int chunk, const int32_t *cu_seqlens, void *stream);

/*
 * gla_chunk_fwd_noalloc — gla_chunk_fwd for callers that may not allocate device memory.
 *
 * The pages describe no counterpart of this entry point; it exists for callers
 * that cannot let a library allocate: a host whose memory manager owns the
 * whole device pool and forbids other allocations, a serving loop with a fixed
 * memory budget where an allocation could fail or stall at the wrong time, or a
 * plugin host that only hands its plugins the input and output buffers.
 *
 * Arguments, results and errors are those of gla_chunk_fwd, computed with the
 * same schedule.  The difference: when that schedule splits long sequences
 * into segments, the segment states live in a scratch array that is part of
 * the library's device image (GLA_NOALLOC_SCRATCH_BYTES bytes, reserved on
 * every device that loads the library, until the process exits) instead of
 * memory taken with cudaMallocAsync.  The call itself never allocates or frees
 * device memory.  A problem whose segment states need more than that array is
 * rejected with GLA_ERR_SCRATCH_LIMIT before anything is launched.  The
 * segment states take 2 * chains * (nseg - 1) * dk * dv * 4 bytes, where
 * chains = B * H and the schedule keeps chains * nseg <= SMs, so at most
 * 2 * (SMs - chains) * dk * dv * 4 bytes: every shape the tensor-core kernel
 * takes (largest state 96 x 192) fits on a GB300 (152 SMs), so the limit is
 * never hit there.
 *
 * The array is placed on a device when the library's forward kernels are
 * loaded onto it.  With CUDA's lazy module loading (the default) that is the
 * first call on that device of any entry point using them, not the moment the
 * library is loaded; if that first call is this one and the device has no
 * room left, it returns GLA_ERR_NOMEM (and a later call tries again).  The
 * first call on each device also looks up that device's address of the array
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the one array and every launch overwrites the parts it reads,
 * so nothing carries over between calls, but calls whose work overlaps on the
 * GPU (different streams, or different host threads without ordering) race on
 * it: serialise them.
 */
#define GLA_NOALLOC_SCRATCH_BYTES (24u * 1024u * 1024u)
GLA_API int gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_decay,
                                  const float *h0, void *out, float *hT, int B, int T, int H, int dk,
                                  int dv, int chunk, const int32_t *cu_seqlens, void *stream);

/*
 * gla_chunk_fwd_host — gla_chunk_fwd on HOST arrays, with the copies overlapped.
 *
 * Computes the map of gla_chunk_fwd (same recurrence, same kernels) for a
 * dense batch whose q, k, v, log_decay and h0 live in host memory, and writes
 * out and hT to host memory.  The work is cut into at most 8 groups, none
 * under 8 MiB of copies unless the batch is smaller: groups of whole
 * sequences, or, when that makes more groups (few, long sequences), ranges of
 * whole chunks of rows of every sequence, each computed from the state the
 * previous range left.  Group g+1 is copied to the device while group g
 * computes on `stream` and group g-1 is copied back on a third (the
 * library's own), so the copies in both directions and the compute run at the
 * same time.  A group is computed as a gla_chunk_fwd call of its own, so
 * results can differ from one gla_chunk_fwd call on the whole batch in the
 * last bits (the schedule depends on the number of chains and chunks), never
 * by more than rounding.
 *
 * Arguments are those of gla_chunk_fwd without cu_seqlens (packed batches are
 * not taken here), with every array a HOST pointer in the same layout:
 *   q, k [B, T, H, dk] bf16; v, out [B, T, H, dv] bf16; log_decay [H] f32;
 *   h0, hT [B, H, dk, dv] f32 or NULL.
 * Page-locked (pinned) host memory lets the copies run asynchronously and
 * overlap; pageable memory works but the driver stages it and the overlap is
 * lost.  No host alignment is required.
 *
 * Ownership: the arrays stay the caller's.  The call enqueues work and returns;
 * out and hT are written, and the input arrays may be reused, once `stream`
 * reaches the point of the call (cudaStreamSynchronize(stream) or an event
 * recorded after the call).  Device scratch for two groups plus log_decay is
 * taken with cudaMallocAsync on `stream` and freed in stream order.  The two
 * copy streams are the library's own (per device, created on first use).
 *
 * Errors: GLA_ERR_ARG / GLA_ERR_UNSUPPORTED as gla_chunk_fwd (checked before
 * anything is enqueued); GLA_ERR_NOMEM if the scratch cannot be allocated;
 * GLA_ERR_LAUNCH if an enqueue fails (the call then waits for what it had
 * enqueued before it frees the scratch).  Device-side status as gla_chunk_fwd.
 */
GLA_API int gla_chunk_fwd_host(const void *q, const void *k, const void *v, const float *log_decay,
                               const float *h0, void *out, float *hT, int B, int T, int H, int dk, int dv,
                               int chunk, void *stream);

/* gla_chunk_fwd_f32 — as gla_chunk_fwd with f32 q, k, v and out.  Always runs
 * the SIMT kernel (f32 FMA, no tensor cores): chunk in {16, 32, 64, 128}.
 * The SIMT kernel processes a chunk whose tiles do not fit in shared memory
 * (large dk) as sub-chunks of half the length; the result is the same map. */
GLA_API int gla_chunk_fwd_f32(const float *q, const float *k, const float *v, const float *log_decay,
                      const float *h0, float *out, float *hT, int B, int T, int H, int dk, int dv,
                      int chunk, const int32_t *cu_seqlens, void *stream);

/*
 * gla_chunk_bwd — gradients of the chunked forward, for training (page
 * "线性注意力模型如何实现固定推理状态", section "挑战 3": the backward pass
 * differentiates every sequential state update; the page prints no formulas,
 * so these are the chain rule of the recurrence).  With
 *     L = sum(dout .* out) + sum(dhT .* hT),   G_t = dL/dS_t:
 *     G_T = dhT + q_T^T do_T,   G_t = lambda_h G_{t+1} + q_t^T do_t
 *     dq_t = do_t S_t^T,   dk_t = v_t G_t^T,   dv_t = k_t G_t,   dh0 = lambda_h G_1
 * (S_t the forward states).  Each of dv, dk and dq is a chunked recurrence of
 * the same form as the forward: dv and dk walk each sequence backwards in time
 * (from the state dhT), dq forwards (from h0); three launches in all.
 *
 *   q, k         [B, T, H, dk] bf16 (packed [1, T, H, dk] with cu_seqlens)
 *   v, dout      [B, T, H, dv] bf16
 *   log_decay    [H] f32
 *   h0           [B|N, H, dk, dv] f32 or NULL (zeros), as in the forward
 *   dhT          [B|N, H, dk, dv] f32 or NULL (zeros): gradient with respect to hT
 *   dq, dk       [B, T, H, dk] bf16, written
 *   dv           [B, T, H, dv] bf16, written
 *   dh0          [B|N, H, dk, dv] f32, written; NULL to skip
 *   B, T, H, dk, dv, chunk, cu_seqlens, stream: as gla_chunk_fwd
 * With chunk == 128, 32 | dk <= 128, 64 | dv <= 192 and dv + 2 dk <= 384 it
 * runs on the tensor cores: two state passes (S before every chunk from h0,
 * forwards; the gradient state G at every chunk's end from dhT, backwards;
 * both kept as bf16 tiles in stream-ordered scratch of 2 x 2 dk dv bytes per
 * chunk, GLA_ERR_NOMEM if it cannot be had) and one kernel over all (chunk,
 * head) pairs at once.  Heads with log_decay < -0.3, and every other shape or
 * chunk in {16, 32, 64}, run three chunked recurrences on the SIMT kernel
 * (f32 accumulation; dv and dk backwards in time from dhT, dq forwards from
 * h0).  No pointer may alias another.  Returns a gla_status.
 */
GLA_API int gla_chunk_bwd(const void *q, const void *k, const void *v, const void *dout, const float *log_decay,
                          const float *h0, const float *dhT, void *dq, void *dk_out, void *dv_out, float *dh0,
                          int B, int T, int H, int dk, int dv, int chunk, const int32_t *cu_seqlens,
                          void *stream);

/*
 * Training with saved states.  The tensor-core backward begins by walking
 * every chain forwards to recover the state before each chunk (it reads k and
 * v again); the forward already holds that state, as the bf16 tile its
 * inter-chunk product reads.  gla_chunk_fwd_save is gla_chunk_fwd that also
 * writes those tiles out, and gla_chunk_bwd_saved is gla_chunk_bwd that takes
 * them and skips its forward walk.
 *
 * gla_state_images_bytes — bytes of the state-image buffer for a batch:
 *     (rows / 128 + B + 1) * H * dk * dv * 2,   rows = B * T (dense) or T
 *     (packed: B sequences, T total rows);
 * chunk c of sequence s (first row start_s) is the dk x dv bf16 tile at slot
 * start_s / 128 + s + c, the state in force before the chunk (h0, or zeros,
 * for c = 0), stored in the kernels' shared-memory layout (dv in 64-column
 * atoms of dk rows x 128 bytes, the 16-byte pieces of row r permuted by
 * r mod 8): treat it as opaque.  Slots between sequences are never written.
 * Returns 0 for invalid sizes.
 */
GLA_API long long gla_state_images_bytes(int B, int T, int H, int dk, int dv, int packed);

/*
 * gla_chunk_fwd_save — as gla_chunk_fwd (same arguments, same out and hT)
 * plus state_images: a device buffer of gla_state_images_bytes(...) bytes,
 * 16-byte aligned, written as described above.  Only where both the forward
 * and the backward run on the tensor cores: chunk == 128, 32 | dk <= 128,
 * 64 | dv <= 192, dv + 2 dk <= 384; otherwise GLA_ERR_UNSUPPORTED (use
 * gla_chunk_fwd and gla_chunk_bwd).  Extra traffic: 2 dk dv bytes per chunk
 * and head written.
 */
GLA_API int gla_chunk_fwd_save(const void *q, const void *k, const void *v, const float *log_decay,
                               const float *h0, void *out, float *hT, void *state_images, int B, int T, int H,
                               int dk, int dv, int chunk, const int32_t *cu_seqlens, void *stream);

/*
 * gla_chunk_bwd_saved — as gla_chunk_bwd, with state_images as written by
 * gla_chunk_fwd_save for the same q, k, v, log_decay, h0, sizes and
 * cu_seqlens (read only).  Scratch: one image array (the gradient states)
 * instead of two.  Same support rule and errors as gla_chunk_fwd_save.
 */
GLA_API int gla_chunk_bwd_saved(const void *q, const void *k, const void *v, const void *dout,
                                const float *log_decay, const float *h0, const float *dhT,
                                const void *state_images, void *dq, void *dk_out, void *dv_out, float *dh0, int B,
                                int T, int H, int dk, int dv, int chunk, const int32_t *cu_seqlens, void *stream);

/* gla_chunk_bwd_f32 — as gla_chunk_bwd with f32 q, k, v, dout, dq, dk_out, dv_out. */
GLA_API int gla_chunk_bwd_f32(const float *q, const float *k, const float *v, const float *dout,
                              const float *log_decay, const float *h0, const float *dhT, float *dq,
                              float *dk_out, float *dv_out, float *dh0, int B, int T, int H, int dk, int dv,
                              int chunk, const int32_t *cu_seqlens, void *stream);

/*
 * gla_decode_step — one recurrent decode step for N independent sequences
 * (page "线性注意力模型如何实现固定推理状态", section "i14 与 Laplace 3B 架构":
 * O(1) work per generated token with a fixed-size state; section "Trainium2 上的
 * 推理优化": one fixed state page per sequence):
 *     state <- lambda_h * state + k^T v      (in place)
 *     out    = q state                        (with the updated state)
 *
 *   q, k         [N, H, dk] bf16
 *   v            [N, H, dv] bf16
 *   log_decay    [H] f32
 *   state_inout  [N, H, dk, dv] f32, read and written once
 *   out          [N, H, dv] bf16, written
 *   N, H > 0; 1 <= dk <= 256; 4 <= dv <= 1024 with dv % 4 == 0
 *   stream       cudaStream_t
 * Returns a gla_status.
 */
GLA_API int gla_decode_step(const void *q, const void *k, const void *v, const float *log_decay,
                    float *state_inout, void *out, int N, int H, int dk, int dv, void *stream);

/* gla_decode_step_f32 — as gla_decode_step with f32 q, k, v and out. */
GLA_API int gla_decode_step_f32(const float *q, const float *k, const float *v, const float *log_decay,
                        float *state_inout, float *out, int N, int H, int dk, int dv, void *stream);

/*
 * gla_decode_step_paged — gla_decode_step with the states kept in a pool of
 * fixed pages, one page per sequence (page "线性注意力模型如何实现固定推理状态",
 * section "Trainium2 上的推理优化": the serving engine hands every sequence a
 * fixed state page in its pool; each new decode batch width cost a separate
 * compiled shape, so batches were padded to fixed widths).  Row n of the batch
 * uses page slots[n]:
 *     S = state_pool[slots[n]]:  S <- lambda_h S + k^T v;  out[n] = q S
 * A negative slot marks a padding row: its out row is written as zeros and no
 * page is touched.  Any N runs with the same kernel; a padded fixed-width call
 * makes no allocation or host synchronisation, so it can be captured in a
 * CUDA graph and replayed after rewriting `slots` (and q, k, v) in place.
 *
 *   q, k, v, out, log_decay, N, H, dk, dv: as gla_decode_step (bf16)
 *   state_pool   [nslots, H, dk, dv] f32, pages read and written in place
 *   slots        [N] int32 on the device; each slot < nslots or negative
 *   nslots       pages in the pool (> 0)
 * Two rows must not name the same page (their updates would race).  A slot
 * >= nslots is a device-side error: the row is treated as padding and
 * GLA_ERR_DEVICE_ARG is recorded for gla_last_device_status.
 */
GLA_API int gla_decode_step_paged(const void *q, const void *k, const void *v, const float *log_decay,
                                  float *state_pool, const int32_t *slots, int nslots, void *out, int N, int H,
                                  int dk, int dv, void *stream);

/*
 * gla_decode_step_gated / gla_decode_step_paged_gated — the decode steps with the output gate fused
 * into the write of out: out[n, h, :] = (q S)[:] * f(g[n, h, :]), f per gate_kind (gla_gate_kind).  The
 * state update is unchanged.  A padding row of the paged form still writes zeros.
 *   g          [N, H, dv] bf16, the layout of out; device, 16-byte aligned; read only
 *   gate_kind  GLA_GATE_SILU or GLA_GATE_SIGMOID (else GLA_ERR_ARG)
 *   the other arguments and errors: as gla_decode_step / gla_decode_step_paged.
 */
/*
 * gla_decode_step_layers — decode steps of L layers at once over pages that hold every layer of a
 * sequence (page "线性注意力模型如何实现固定推理状态", section "Trainium2 上的推理优化": the serving
 * engine gives each sequence one fixed state page for the whole model, and every new batch width cost
 * a separately compiled shape).  Pages are [page_layers, H, dk, dv] f32; row n of the batch uses page
 * slots[n], and layer l (0 <= l < L) of the call updates and reads layer layer0 + l of it:
 *     S = state_pool[slots[n], layer0 + l, h]:  S <- lambda_{l,h} S + k^T v;  out[l, n, h] = q S
 * (times the output gate's factor when g is given).  One launch covers L * N * H chains with the same
 * kernel for any L and N.  A model whose layer l + 1 needs layer l's output calls it once per layer
 * (L = 1, layer0 = l); L > 1 serves inputs of several layers that are ready together.
 *   q, k         [L, N, H, dk] bf16;  v, out [L, N, H, dv] bf16
 *   g            [L, N, H, dv] bf16 or NULL (no gate);  gate_kind as gla_chunk_fwd_gated when g is given
 *   log_decay    [L, H] f32: the decays of layers layer0 .. layer0 + L - 1
 *   state_pool   [nslots, page_layers, H, dk, dv] f32, read and written in place
 *   slots        [N] int32 on the device; negative: a padding row (zero out, no page touched)
 *   0 <= layer0, layer0 + L <= page_layers (else GLA_ERR_ARG); pointers 16-byte aligned; as
 *   gla_decode_step_paged otherwise (two rows must not name the same page).
 */
GLA_API int gla_decode_step_layers(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                                   const float *log_decay, float *state_pool, const int32_t *slots, int nslots,
                                   int page_layers, int layer0, int L, void *out, int N, int H, int dk, int dv,
                                   void *stream);

GLA_API int gla_decode_step_gated(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                                  const float *log_decay, float *state_inout, void *out, int N, int H, int dk,
                                  int dv, void *stream);
GLA_API int gla_decode_step_paged_gated(const void *q, const void *k, const void *v, const void *g,
                                        int gate_kind, const float *log_decay, float *state_pool,
                                        const int32_t *slots, int nslots, void *out, int N, int H, int dk,
                                        int dv, void *stream);

/*
 * gla_conv1d_silu — causal depthwise Conv1d of width 4 followed by SiLU, per
 * channel (page "线性注意力模型如何实现固定推理状态", section "i14 与 Laplace 3B
 * 架构", "归一化与卷积": a 4-token per-channel summary of the normalised
 * residual stream ahead of the QKVG projection; the page prints no formula,
 * this is the plain reading).  For channel c at token t of a sequence:
 *     z = bias[c] + sum_{k=0..3} weight[c][k] x_{t-3+k}[c]   (weight[c][3] meets x_t)
 *     y_t[c] = z * sigmoid(z)
 * The three inputs before a sequence's first token come from state_in (oldest
 * first), or are zero; state_out receives each sequence's last three inputs
 * (for a sequence shorter than three, the newest of state_in fill the front).
 *
 *   x, y         [B, T, D] bf16 (packed [1, T, D] with cu_seqlens, and then B
 *                is the number of sequences N; rows past cu_seqlens[N] are
 *                never written, though tiles that reach into them may read them)
 *   weight       [D, 4] f32;  bias [D] f32 or NULL
 *   state_in     [B|N, D, 3] f32 or NULL (zeros);  state_out [B|N, D, 3] f32 or NULL
 *   D % 8 == 0; every pointer 16-byte aligned.  Memory-bound: x is read and y
 *   written once.  Returns a gla_status.
 */
GLA_API int gla_conv1d_silu(const void *x, const float *weight, const float *bias, const float *state_in,
                            float *state_out, void *y, int B, int T, int D, const int32_t *cu_seqlens,
                            void *stream);

/* gla_conv1d_silu_f32 — as gla_conv1d_silu with f32 x and y. */
GLA_API int gla_conv1d_silu_f32(const float *x, const float *weight, const float *bias, const float *state_in,
                                float *state_out, float *y, int B, int T, int D, const int32_t *cu_seqlens,
                                void *stream);

/*
 * gla_conv1d_silu_step — the same operation for one new token of N sequences,
 * in place on their conv states (decode):
 *     y[n] = SiLU(bias + w0 s0 + w1 s1 + w2 s2 + w3 x[n]);  state[n] <- (s1, s2, x[n])
 *   x, y [N, D] bf16;  state_inout [N, D, 3] f32;  weight, bias as above.
 */
GLA_API int gla_conv1d_silu_step(const void *x, const float *weight, const float *bias, float *state_inout,
                                 void *y, int N, int D, void *stream);

/*
 * gla_last_device_status — synchronise `stream`, then return and clear the
 * device status word: GLA_OK, GLA_ERR_TIMEOUT or GLA_ERR_DEVICE_ARG for the
 * first failure recorded by any kernel of this library on the current device
 * since the previous call.  Returns GLA_ERR_LAUNCH if synchronisation fails.
 */
GLA_API int gla_last_device_status(void *stream);

/*
 * gla_chunk_kernel — which kernel a chunked entry point runs for these sizes on
 * the current device (a host-side query; launches nothing).
 *   op     GLA_OP_FORWARD (gla_chunk_fwd and its _noalloc, _host and _save
 *          forms), GLA_OP_FORWARD_GATED (gla_chunk_fwd_gated) or GLA_OP_BACKWARD
 *          (gla_chunk_bwd); else GLA_ERR_ARG
 *   dtype  GLA_BF16 (the bf16 entry points) or GLA_F32 (the _f32 ones)
 *   dk, dv, chunk  as the entry point would get them
 * Returns GLA_KERNEL_TENSOR_CORE, GLA_KERNEL_SIMT, or a negative gla_status
 * for sizes the entry point rejects (GLA_ERR_UNSUPPORTED, also on a device
 * that is not sm_103).
 *
 * The tensor-core kernels (tcgen05 MMAs with TMEM accumulators, fed by TMA)
 * take bf16 inputs with chunk 128 or 64, dk a multiple of 32 up to 128 and dv
 * a multiple of 64 up to 192 whose tiles fit in shared memory: every such
 * shape but dk 128 with dv 192, which needs 240 KB for the forward's two Q, K
 * and V tiles against the 227 KB a block may use (the gated forward needs
 * 16 KB more; the backward also needs dv + 2 dk <= 384).  A chunk of 64 runs
 * as two 64-token chunks per 128-row tile: the second chunk's carried-state
 * term through the first chunk's keys and values is the tile's lower-left
 * attention block, which is the chunk-64 recurrence without rounding the
 * state between the two chunks to bf16 (the same map up to rounding).  Every
 * other case runs the f32-FMA SIMT kernel, which is correct for all of them
 * but about ten times slower on the shapes both kernels take.
 */
typedef enum { GLA_OP_FORWARD = 0, GLA_OP_FORWARD_GATED = 1, GLA_OP_BACKWARD = 2 } gla_op;
typedef enum { GLA_BF16 = 0, GLA_F32 = 1 } gla_dtype;
typedef enum { GLA_KERNEL_TENSOR_CORE = 1, GLA_KERNEL_SIMT = 2 } gla_kernel_kind;
GLA_API int gla_chunk_kernel(int op, int dtype, int dk, int dv, int chunk);

/* gla_status_str — static, NUL-terminated description of a gla_status value. */
GLA_API const char *gla_status_str(int status);

/* gla_kernel_launches — number of CUDA kernels this library has launched in
 * this process (all devices, all threads), counted on the host at launch. */
GLA_API uint64_t gla_kernel_launches(void);

/* gla_version — library version as major*10000 + minor*100 + patch. */
GLA_API int gla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GLA_H_ */
