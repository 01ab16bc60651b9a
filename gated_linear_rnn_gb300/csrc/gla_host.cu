// gla_host.cu — the chunked forward on host-resident arrays, with the copies overlapped.
//
// For callers whose q, k, v live in (pinned) host memory and who want out and hT back there: the
// work is cut into groups; each group's host-to-device copies (one library stream), its forward (the
// caller's stream) and its device-to-host copies (another library stream) are ordered by events, so
// that group g+1 is copied in while group g computes and group g-1 is copied out.  Two device slots
// hold the groups in flight; they come from stream-ordered scratch on the caller's stream.
// Sequences of at least two chunks are cut in time: a group is a chunk-aligned range of rows of every
// sequence (one strided 2-D copy per array), computed with the state left by the previous range as its
// initial state (the recurrence carries nothing else across a chunk boundary), so the first copy-in and
// the last compute and copy-out, which nothing overlaps, are a small part of the whole.  Shorter
// sequences are grouped whole.  Host code only: the computation is gla_chunk_fwd's.
#include <mutex>

#include "gla_common.cuh"

namespace gla {

int tc_chunk_fwd_bf16(const void *, const void *, const void *, const float *, const float *, void *, float *, int,
                      int, int, int, int, const int32_t *, cudaStream_t);
int simt_chunk_fwd_bf16(const void *, const void *, const void *, const float *, const float *, void *, float *, int,
                        int, int, int, int, int, const int32_t *, cudaStream_t);
bool tc_chunk_supported(int dk, int dv, int chunk);
bool tc_chunk_len(int chunk);

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 8;  // groups of whole sequences, or time ranges (16 ranges were no faster)
constexpr size_t kMinGroupBytes = size_t(8) << 20;

// Copy streams of a device, created once and kept for the process: one per direction.  (Splitting
// each copy over two streams per direction was slower on GB300 in this pipeline: the two directions
// share the host link, 1.10 ms for this layer's 201 MB in and 110 MB out run at once against 0.97 ms
// for the input alone.)
struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaError_t err = cudaSuccess;
};
std::once_flag g_streams_once[kMaxDevices];
CopyStreams g_streams[kMaxDevices];

const CopyStreams *copy_streams() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_streams_once[dev], [dev]() {
        CopyStreams &c = g_streams[dev];
        c.err = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking);
        if (c.err == cudaSuccess) c.err = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking);
    });
    return g_streams[dev].err == cudaSuccess ? &g_streams[dev] : nullptr;
}

int forward_on_device(const void *qd, const void *kd, const void *vd, const float *ld_d, const float *h0d,
                      void *od, float *hTd, int nseq, int T, int H, int dk, int dv, int chunk, cudaStream_t st) {
    return (tc_chunk_len(chunk) && tc_chunk_supported(dk, dv, 128))
               ? tc_chunk_fwd_bf16(qd, kd, vd, ld_d, h0d, od, hTd, nseq, T, H, dk, dv, nullptr, st)
               : simt_chunk_fwd_bf16(qd, kd, vd, ld_d, h0d, od, hTd, nseq, T, H, dk, dv, chunk, nullptr, st);
}

// B blocks of `width` bytes at pitches dpitch and spitch: one 2-D copy when the pitches are within the
// device's limit, else one copy per block.
bool copy_blocks(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, int B, cudaMemcpyKind kind,
                 size_t max_pitch, cudaStream_t s) {
    if (dpitch <= max_pitch && spitch <= max_pitch)
        return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, (size_t)B, kind, s) == cudaSuccess;
    for (int b = 0; b < B; ++b)
        if (cudaMemcpyAsync(static_cast<uint8_t *>(dst) + (size_t)b * dpitch,
                            static_cast<const uint8_t *>(src) + (size_t)b * spitch, width, kind, s) != cudaSuccess)
            return false;
    return true;
}

// Time ranges of `rows` rows (a multiple of the chunk; the last may be short) over all B sequences.
// Device: two slots of [B, rows, H, d] for q, k, v and out, and two state buffers [B, H, dk, dv]: range
// g starts from buffer (g + 1) % 2 (the caller's h0 is copied there for range 0) and leaves its final
// state in buffer g % 2.
int host_time_ranges(const void *q, const void *k, const void *v, const float *log_decay, const float *h0, void *out,
                     float *hT, int B, int T, int H, int dk, int dv, int chunk, int rows, int nranges,
                     const CopyStreams *cs, cudaStream_t st) {
    const size_t qk_r = (size_t)H * dk * 2, vo_r = (size_t)H * dv * 2;  // bytes per (sequence, row)
    const size_t st_b = (size_t)B * H * dk * dv * 4;
    const size_t slot_b = (size_t)B * rows * (2 * qk_r + 2 * vo_r);
    const size_t ld_b = ((size_t)H * 4 + 255) / 256 * 256;
    uint8_t *ws = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&ws), 2 * slot_b + 2 * st_b + ld_b, st) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_NOMEM;
    }
    float *state[2] = {reinterpret_cast<float *>(ws + 2 * slot_b), reinterpret_cast<float *>(ws + 2 * slot_b + st_b)};
    float *ld_d = reinterpret_cast<float *>(ws + 2 * slot_b + 2 * st_b);
    int dev = 0, pitch_attr = 0;
    size_t max_pitch = 0;  // 0: every copy goes block by block
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&pitch_attr, cudaDevAttrMaxPitch, dev) == cudaSuccess)
        max_pitch = (size_t)(unsigned)pitch_attr;
    else
        cudaGetLastError();
    constexpr int kEvPerRange = 3;
    cudaEvent_t ev[kEvPerRange * kMaxGroups + 1];
    int nev = 0, rc = GLA_OK;
    for (; nev < kEvPerRange * nranges + 1; ++nev)
        if (cudaEventCreateWithFlags(&ev[nev], cudaEventDisableTiming) != cudaSuccess) {
            rc = GLA_ERR_LAUNCH;
            break;
        }
    cudaEvent_t *ev_in = ev, *ev_c = ev + nranges, *ev_out = ev + 2 * nranges, ev_start = ev[kEvPerRange * nranges];
    // the copies start after everything already queued on the caller's stream (incl. the workspace)
    if (rc == GLA_OK && (cudaEventRecord(ev_start, st) != cudaSuccess ||
                         cudaStreamWaitEvent(cs->in, ev_start, 0) != cudaSuccess))
        rc = GLA_ERR_LAUNCH;
    if (rc == GLA_OK && cudaMemcpyAsync(ld_d, log_decay, (size_t)H * 4, cudaMemcpyHostToDevice, cs->in) != cudaSuccess)
        rc = GLA_ERR_LAUNCH;
    if (rc == GLA_OK && h0 && cudaMemcpyAsync(state[1], h0, st_b, cudaMemcpyHostToDevice, cs->in) != cudaSuccess)
        rc = GLA_ERR_LAUNCH;
    for (int g = 0; g < nranges && rc == GLA_OK; ++g) {
        const int t0 = g * rows, n = (T - t0 < rows) ? T - t0 : rows;
        uint8_t *qd = ws + (size_t)(g & 1) * slot_b, *kd = qd + (size_t)B * rows * qk_r;
        uint8_t *vd = kd + (size_t)B * rows * qk_r, *od = vd + (size_t)B * rows * vo_r;
        // in: the slot is free once range g-2 has been copied out; each array is B strided blocks
        if (g >= 2 && cudaStreamWaitEvent(cs->in, ev_out[g - 2], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK &&
            (!copy_blocks(qd, n * qk_r, static_cast<const uint8_t *>(q) + t0 * qk_r, (size_t)T * qk_r, n * qk_r, B,
                          cudaMemcpyHostToDevice, max_pitch, cs->in) ||
             !copy_blocks(kd, n * qk_r, static_cast<const uint8_t *>(k) + t0 * qk_r, (size_t)T * qk_r, n * qk_r, B,
                          cudaMemcpyHostToDevice, max_pitch, cs->in) ||
             !copy_blocks(vd, n * vo_r, static_cast<const uint8_t *>(v) + t0 * vo_r, (size_t)T * vo_r, n * vo_r, B,
                          cudaMemcpyHostToDevice, max_pitch, cs->in) ||
             cudaEventRecord(ev_in[g], cs->in) != cudaSuccess))
            rc = GLA_ERR_LAUNCH;
        // compute on the caller's stream, from the state the previous range left
        if (rc == GLA_OK && cudaStreamWaitEvent(st, ev_in[g], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK) {
            const float *h0d = (g == 0 && h0 == nullptr) ? nullptr : state[(g + 1) & 1];
            rc = forward_on_device(qd, kd, vd, ld_d, h0d, od, state[g & 1], B, n, H, dk, dv, chunk, st);
        }
        if (rc == GLA_OK && cudaEventRecord(ev_c[g], st) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        // out
        if (rc == GLA_OK && cudaStreamWaitEvent(cs->out, ev_c[g], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK &&
            (!copy_blocks(static_cast<uint8_t *>(out) + t0 * vo_r, (size_t)T * vo_r, od, n * vo_r, n * vo_r, B,
                          cudaMemcpyDeviceToHost, max_pitch, cs->out) ||
             (g == nranges - 1 && hT &&
              cudaMemcpyAsync(hT, state[g & 1], st_b, cudaMemcpyDeviceToHost, cs->out) != cudaSuccess) ||
             cudaEventRecord(ev_out[g], cs->out) != cudaSuccess))
            rc = GLA_ERR_LAUNCH;
    }
    // the caller's stream continues after every copy out; the workspace goes back in stream order
    for (int g = 0; g < nranges && rc == GLA_OK; ++g)
        if (cudaStreamWaitEvent(st, ev_out[g], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
    if (rc != GLA_OK) {
        // a failed enqueue may leave copies in flight that no event orders before the free: drain
        // the copy streams and the caller's stream first
        cudaStreamSynchronize(cs->in);
        cudaStreamSynchronize(cs->out);
        cudaStreamSynchronize(st);
        cudaGetLastError();
    }
    cudaFreeAsync(ws, st);
    for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);
    return rc;
}

}  // namespace

int chunk_fwd_host_bf16(const void *q, const void *k, const void *v, const float *log_decay, const float *h0,
                        void *out, float *hT, int B, int T, int H, int dk, int dv, int chunk, cudaStream_t st) {
    const CopyStreams *cs = copy_streams();
    if (cs == nullptr) return GLA_ERR_LAUNCH;
    const size_t tok = (size_t)T * H;                  // token-heads per sequence
    const size_t qk_b = tok * dk * 2, vo_b = tok * dv * 2, st_b = (size_t)H * dk * dv * 4;  // bytes per sequence
    // groups of whole sequences: at most 8 of them, and none under kMinGroupBytes of copies unless
    // the batch is that small (each group costs a few launches and events)
    const size_t seq_b = 2 * qk_b + 2 * vo_b + ((h0 ? 1 : 0) + (hT ? 1 : 0)) * st_b;
    int per_group = (B + kMaxGroups - 1) / kMaxGroups;
    const size_t min_seqs = (kMinGroupBytes + seq_b - 1) / seq_b;
    if ((size_t)per_group < min_seqs) per_group = min_seqs < (size_t)B ? (int)min_seqs : B;
    const int ngroups = (B + per_group - 1) / per_group;
    // time ranges of whole chunks, on the same terms: taken when they make more groups (few, long
    // sequences), since every group adds copies and launches
    {
        const int nch = (T + chunk - 1) / chunk;
        const size_t chunk_b = (size_t)B * chunk * H * (2 * dk + 2 * dv) * 2;  // copies of one chunk of rows
        int per = (nch + kMaxGroups - 1) / kMaxGroups;
        const size_t min_per = (kMinGroupBytes + chunk_b - 1) / chunk_b;
        if ((size_t)per < min_per) per = min_per < (size_t)nch ? (int)min_per : nch;
        const int nranges = (nch + per - 1) / per;
        if (nranges > ngroups)
            return host_time_ranges(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, chunk, per * chunk, nranges, cs,
                                    st);
    }
    const size_t slot_b = (size_t)per_group * (2 * qk_b + 2 * vo_b + 2 * st_b);
    const size_t ld_b = ((size_t)H * 4 + 255) / 256 * 256;
    uint8_t *ws = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&ws), 2 * slot_b + ld_b, st) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_NOMEM;
    }
    float *ld_d = reinterpret_cast<float *>(ws + 2 * slot_b);  // the device copy of log_decay
    constexpr int kEvPerGroup = 3;
    cudaEvent_t ev[kEvPerGroup * kMaxGroups + 1];
    int nev = 0, rc = GLA_OK;
    for (; nev < kEvPerGroup * ngroups + 1; ++nev)
        if (cudaEventCreateWithFlags(&ev[nev], cudaEventDisableTiming) != cudaSuccess) {
            rc = GLA_ERR_LAUNCH;
            break;
        }
    cudaEvent_t *ev_in = ev, *ev_c = ev + ngroups, *ev_out = ev + 2 * ngroups, ev_start = ev[kEvPerGroup * ngroups];
    // the copies start after everything already queued on the caller's stream (incl. the workspace)
    if (rc == GLA_OK && (cudaEventRecord(ev_start, st) != cudaSuccess ||
                         cudaStreamWaitEvent(cs->in, ev_start, 0) != cudaSuccess))
        rc = GLA_ERR_LAUNCH;
    if (rc == GLA_OK && cudaMemcpyAsync(ld_d, log_decay, (size_t)H * 4, cudaMemcpyHostToDevice, cs->in) != cudaSuccess)
        rc = GLA_ERR_LAUNCH;
    for (int g = 0; g < ngroups && rc == GLA_OK; ++g) {
        const int b0 = g * per_group, nb = (B - b0 < per_group) ? B - b0 : per_group;
        uint8_t *slot = ws + (size_t)(g & 1) * slot_b;
        uint8_t *qd = slot, *kd = qd + per_group * qk_b, *vd = kd + per_group * qk_b, *od = vd + per_group * vo_b;
        float *h0d = reinterpret_cast<float *>(od + per_group * vo_b), *hTd = h0d + (size_t)per_group * H * dk * dv;
        // in: the slot is free once group g-2 has been copied out
        if (g >= 2 && cudaStreamWaitEvent(cs->in, ev_out[g - 2], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK) {
            const uint8_t *qh = static_cast<const uint8_t *>(q) + b0 * qk_b;
            const uint8_t *kh = static_cast<const uint8_t *>(k) + b0 * qk_b;
            const uint8_t *vh = static_cast<const uint8_t *>(v) + b0 * vo_b;
            if (cudaMemcpyAsync(qd, qh, nb * qk_b, cudaMemcpyHostToDevice, cs->in) != cudaSuccess ||
                cudaMemcpyAsync(kd, kh, nb * qk_b, cudaMemcpyHostToDevice, cs->in) != cudaSuccess ||
                cudaMemcpyAsync(vd, vh, nb * vo_b, cudaMemcpyHostToDevice, cs->in) != cudaSuccess ||
                (h0 && cudaMemcpyAsync(h0d, h0 + (size_t)b0 * H * dk * dv, nb * st_b, cudaMemcpyHostToDevice,
                                       cs->in) != cudaSuccess) ||
                cudaEventRecord(ev_in[g], cs->in) != cudaSuccess)
                rc = GLA_ERR_LAUNCH;
        }
        // compute on the caller's stream
        if (rc == GLA_OK && cudaStreamWaitEvent(st, ev_in[g], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK)
            rc = forward_on_device(qd, kd, vd, ld_d, h0 ? h0d : nullptr, od, hT ? hTd : nullptr, nb, T, H, dk, dv,
                                   chunk, st);
        if (rc == GLA_OK && cudaEventRecord(ev_c[g], st) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        // out
        if (rc == GLA_OK && cudaStreamWaitEvent(cs->out, ev_c[g], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK) {
            if (cudaMemcpyAsync(static_cast<uint8_t *>(out) + b0 * vo_b, od, nb * vo_b, cudaMemcpyDeviceToHost,
                                cs->out) != cudaSuccess ||
                (hT && cudaMemcpyAsync(hT + (size_t)b0 * H * dk * dv, hTd, nb * st_b, cudaMemcpyDeviceToHost,
                                       cs->out) != cudaSuccess) ||
                cudaEventRecord(ev_out[g], cs->out) != cudaSuccess)
                rc = GLA_ERR_LAUNCH;
        }
    }
    // the caller's stream continues after every copy out; the workspace goes back in stream order
    for (int g = 0; g < ngroups && rc == GLA_OK; ++g)
        if (cudaStreamWaitEvent(st, ev_out[g], 0) != cudaSuccess) rc = GLA_ERR_LAUNCH;
    if (rc != GLA_OK) {
        // a failed enqueue may leave copies in flight that no event orders before the free: drain
        // the copy streams and the caller's stream first
        cudaStreamSynchronize(cs->in);
        cudaStreamSynchronize(cs->out);
        cudaStreamSynchronize(st);
        cudaGetLastError();
    }
    cudaFreeAsync(ws, st);
    for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);
    return rc;
}

}  // namespace gla
