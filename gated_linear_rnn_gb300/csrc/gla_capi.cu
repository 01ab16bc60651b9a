// gla_capi.cu — the extern "C" boundary of libgla.so.
//
// Host-side argument checks, the choice between the tensor-core and SIMT
// kernels, and the device status word.  Declarations and the contract of every
// entry point are in include/gla.h.
#include <atomic>
#include <mutex>

#include "gla_common.cuh"

namespace gla {

// kernels (defined in the other translation units)
int simt_chunk_fwd_f32(const float *, const float *, const float *, const float *, const float *, float *,
                       float *, int, int, int, int, int, int, const int32_t *, cudaStream_t);
int simt_chunk_fwd_bf16(const void *, const void *, const void *, const float *, const float *, void *,
                        float *, int, int, int, int, int, int, const int32_t *, cudaStream_t);
int decode_step_bf16(const void *, const void *, const void *, const float *, float *, void *, int, int, int,
                     int, cudaStream_t);
int decode_step_f32(const float *, const float *, const float *, const float *, float *, float *, int, int,
                    int, int, cudaStream_t);
int decode_step_paged_bf16(const void *, const void *, const void *, const float *, float *, const int32_t *, int,
                           void *, int, int, int, int, cudaStream_t);
bool tc_chunk_supported(int dk, int dv, int chunk);
bool tc_gate_supported(int dk, int dv);
int tc_chunk_fwd_bf16(const void *, const void *, const void *, const float *, const float *, void *, float *,
                      int, int, int, int, int, const int32_t *, cudaStream_t);
int tc_chunk_fwd_bf16_noalloc(const void *, const void *, const void *, const float *, const float *, void *,
                              float *, int, int, int, int, int, const int32_t *, cudaStream_t);
int simt_chunk_bwd_f32(const float *, const float *, const float *, const float *, const float *, const float *,
                       const float *, float *, float *, float *, float *, int, int, int, int, int, int,
                       const int32_t *, cudaStream_t);
int simt_chunk_bwd_bf16(const void *, const void *, const void *, const void *, const float *, const float *,
                        const float *, void *, void *, void *, float *, int, int, int, int, int, int,
                        const int32_t *, cudaStream_t);
bool tc_bwd_supported(int dk, int dv, int chunk);
int tc_chunk_bwd_bf16(const void *, const void *, const void *, const void *, const float *, const float *,
                      const float *, void *, void *, void *, float *, int, int, int, int, int, const int32_t *,
                      cudaStream_t);
int tc_chunk_fwd_bf16_save(const void *, const void *, const void *, const float *, const float *, void *, float *,
                           void *, int, int, int, int, int, const int32_t *, cudaStream_t);
int tc_chunk_bwd_bf16_saved(const void *, const void *, const void *, const void *, const float *, const float *,
                            const float *, const void *, void *, void *, void *, float *, int, int, int, int, int,
                            const int32_t *, cudaStream_t);
int conv1d_silu_bf16(const void *, const float *, const float *, const float *, float *, void *, int, int, int,
                     const int32_t *, cudaStream_t);
int conv1d_silu_f32(const float *, const float *, const float *, const float *, float *, float *, int, int, int,
                    const int32_t *, cudaStream_t);
int conv1d_silu_step_bf16(const void *, const float *, const float *, float *, void *, int, int, cudaStream_t);
int chunk_fwd_host_bf16(const void *, const void *, const void *, const float *, const float *, void *, float *,
                        int, int, int, int, int, int, cudaStream_t);
int tc_chunk_fwd_gated_bf16(const void *, const void *, const void *, const void *, int, const float *, const float *,
                            void *, float *, int, int, int, int, int, const int32_t *, cudaStream_t);
int simt_chunk_fwd_gated_bf16(const void *, const void *, const void *, const void *, int, const float *,
                              const float *, void *, float *, int, int, int, int, int, int, const int32_t *,
                              cudaStream_t);
int decode_step_gated_bf16(const void *, const void *, const void *, const void *, int, const float *, float *,
                           const int32_t *, int, void *, int, int, int, int, cudaStream_t);
int decode_step_layers_bf16(const void *, const void *, const void *, const void *, int, const float *, float *,
                            const int32_t *, int, int, int, int, void *, int, int, int, int, cudaStream_t);
int take_status_conv(cudaStream_t);
int take_status_simt(cudaStream_t);
int take_status_bwd(cudaStream_t);
int take_status_decode(cudaStream_t);
int take_status_tc(cudaStream_t);

namespace {
std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
}  // namespace

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

const DeviceInfo &device_info() {
    static DeviceInfo none = {0, 0, 0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return none;
    std::call_once(g_once[dev], [dev]() {
        DeviceInfo d = {0, 0, 0};
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        d.ok = (major == 10 && minor == 3) ? 1 : 0;
        g_info[dev] = d;
    });
    return g_info[dev];
}

// Chunk lengths the tensor-core kernels serve: 128, and 64 as two 64-token chunks per 128-row tile.  In
// such a tile the second chunk's carried-state term through the first chunk's keys and values is the
// tile's lower-left attention block, i.e. the chunk-64 recurrence without rounding the state between the
// two chunks to bf16: the same map up to rounding.
bool tc_chunk_len(int chunk) { return chunk == 64 || chunk == 128; }

namespace {

int check_decays_and_sizes(const float *log_decay, int B, int T, int H, int dk, int dv) {
    if (log_decay == nullptr) return GLA_ERR_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0) return GLA_ERR_ARG;
    return GLA_OK;
}

int check_prefill(const void *q, const void *k, const void *v, const float *ld, const float *h0, const void *out,
                  const float *hT, int B, int T, int H, int dk, int dv, const int32_t *cu) {
    if (!q || !k || !v || !out) return GLA_ERR_ARG;
    int rc = check_decays_and_sizes(ld, B, T, H, dk, dv);
    if (rc) return rc;
    if (dk < 16 || dk > 256 || dv < 16 || dv > 512 || dk % 8 || dv % 8) return GLA_ERR_UNSUPPORTED;
    if ((long long)B * T * H > (1LL << 40)) return GLA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(h0) ||
        !aligned16(hT) || !aligned16(ld) || !aligned16(cu))
        return GLA_ERR_ALIGN;
    if (!device_info().ok) return GLA_ERR_UNSUPPORTED;
    return GLA_OK;
}

int check_backward(const void *q, const void *k, const void *v, const void *dout, const float *ld,
                   const float *h0, const float *dhT, const void *dq, const void *dk, const void *dv,
                   const float *dh0, int B, int T, int H, int dkk, int dvv, const int32_t *cu) {
    if (!dout || !dq || !dk || !dv) return GLA_ERR_ARG;
    int rc = check_prefill(q, k, v, ld, h0, dout, nullptr, B, T, H, dkk, dvv, cu);
    if (rc) return rc;
    if (!aligned16(dhT) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dh0))
        return GLA_ERR_ALIGN;
    return GLA_OK;
}

int check_conv(const void *x, const float *w, const float *b, const float *s_in, const float *s_out, const void *y,
               int B, int T, int D) {
    if (!x || !w || !y) return GLA_ERR_ARG;
    if (B <= 0 || T <= 0 || D <= 0) return GLA_ERR_ARG;
    if (D % 8) return GLA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(b) || !aligned16(s_in) || !aligned16(s_out) || !aligned16(y))
        return GLA_ERR_ALIGN;
    if (!device_info().ok) return GLA_ERR_UNSUPPORTED;
    return GLA_OK;
}

int check_decode(const void *q, const void *k, const void *v, const float *ld, const float *state,
                 const void *out, int N, int H, int dk, int dv) {
    if (!q || !k || !v || !out || !state) return GLA_ERR_ARG;
    int rc = check_decays_and_sizes(ld, N, 1, H, dk, dv);
    if (rc) return rc;
    if (dk > 256 || dv < 4 || dv > 1024 || dv % 4) return GLA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(state) ||
        !aligned16(ld))
        return GLA_ERR_ALIGN;
    if (!device_info().ok) return GLA_ERR_UNSUPPORTED;
    return GLA_OK;
}

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" {

int gla_chunk_fwd(const void *q, const void *k, const void *v, const float *log_decay, const float *h0,
                  void *out, float *hT, int B, int T, int H, int dk, int dv, int chunk,
                  const int32_t *cu_seqlens, void *stream) {
    int rc = check_prefill(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (tc_chunk_len(chunk) && tc_chunk_supported(dk, dv, 128))
        return tc_chunk_fwd_bf16(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens, st);
    return simt_chunk_fwd_bf16(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, chunk, cu_seqlens, st);
}

int gla_chunk_fwd_gated(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                        const float *log_decay, const float *h0, void *out, float *hT, int B, int T, int H, int dk,
                        int dv, int chunk, const int32_t *cu_seqlens, void *stream) {
    if (!g) return GLA_ERR_ARG;
    if (gate_kind != GLA_GATE_SILU && gate_kind != GLA_GATE_SIGMOID) return GLA_ERR_ARG;
    int rc = check_prefill(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    if (!aligned16(g)) return GLA_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    if (tc_chunk_len(chunk) && tc_gate_supported(dk, dv))
        return tc_chunk_fwd_gated_bf16(q, k, v, g, gate_kind, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens,
                                       st);
    return simt_chunk_fwd_gated_bf16(q, k, v, g, gate_kind, log_decay, h0, out, hT, B, T, H, dk, dv, chunk,
                                     cu_seqlens, st);
}

int gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_decay, const float *h0,
                          void *out, float *hT, int B, int T, int H, int dk, int dv, int chunk,
                          const int32_t *cu_seqlens, void *stream) {
    int rc = check_prefill(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (tc_chunk_len(chunk) && tc_chunk_supported(dk, dv, 128))
        return tc_chunk_fwd_bf16_noalloc(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens, st);
    // the SIMT kernel takes no scratch
    return simt_chunk_fwd_bf16(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, chunk, cu_seqlens, st);
}

int gla_chunk_fwd_host(const void *q, const void *k, const void *v, const float *log_decay, const float *h0,
                       void *out, float *hT, int B, int T, int H, int dk, int dv, int chunk, void *stream) {
    // host pointers: the alignment rules of device buffers do not apply (the copies take any address)
    if (!q || !k || !v || !out) return GLA_ERR_ARG;
    int rc = check_decays_and_sizes(log_decay, B, T, H, dk, dv);
    if (rc) return rc;
    if (dk < 16 || dk > 256 || dv < 16 || dv > 512 || dk % 8 || dv % 8) return GLA_ERR_UNSUPPORTED;
    if ((long long)B * T * H > (1LL << 40)) return GLA_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return GLA_ERR_UNSUPPORTED;
    if (!device_info().ok) return GLA_ERR_UNSUPPORTED;
    return chunk_fwd_host_bf16(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, chunk, (cudaStream_t)stream);
}

int gla_chunk_fwd_f32(const float *q, const float *k, const float *v, const float *log_decay, const float *h0,
                      float *out, float *hT, int B, int T, int H, int dk, int dv, int chunk,
                      const int32_t *cu_seqlens, void *stream) {
    int rc = check_prefill(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    return simt_chunk_fwd_f32(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, chunk, cu_seqlens,
                              (cudaStream_t)stream);
}

int gla_chunk_bwd(const void *q, const void *k, const void *v, const void *dout, const float *log_decay,
                  const float *h0, const float *dhT, void *dq, void *dk_out, void *dv_out, float *dh0, int B, int T,
                  int H, int dk, int dv, int chunk, const int32_t *cu_seqlens, void *stream) {
    int rc = check_backward(q, k, v, dout, log_decay, h0, dhT, dq, dk_out, dv_out, dh0, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    if (tc_chunk_len(chunk) && tc_bwd_supported(dk, dv, 128))
        return tc_chunk_bwd_bf16(q, k, v, dout, log_decay, h0, dhT, dq, dk_out, dv_out, dh0, B, T, H, dk, dv,
                                 cu_seqlens, (cudaStream_t)stream);
    return simt_chunk_bwd_bf16(q, k, v, dout, log_decay, h0, dhT, dq, dk_out, dv_out, dh0, B, T, H, dk, dv, chunk,
                               cu_seqlens, (cudaStream_t)stream);
}

long long gla_state_images_bytes(int B, int T, int H, int dk, int dv, int packed) {
    if (B <= 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
    const long long rows = packed ? (long long)T : (long long)B * T;
    return (rows / 128 + B + 1) * (long long)H * dk * dv * 2;
}

int gla_chunk_fwd_save(const void *q, const void *k, const void *v, const float *log_decay, const float *h0,
                       void *out, float *hT, void *state_images, int B, int T, int H, int dk, int dv, int chunk,
                       const int32_t *cu_seqlens, void *stream) {
    int rc = check_prefill(q, k, v, log_decay, h0, out, hT, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    if (!state_images) return GLA_ERR_ARG;
    if (!aligned16(state_images)) return GLA_ERR_ALIGN;
    if (!(tc_chunk_len(chunk) && tc_bwd_supported(dk, dv, 128))) return GLA_ERR_UNSUPPORTED;
    return tc_chunk_fwd_bf16_save(q, k, v, log_decay, h0, out, hT, state_images, B, T, H, dk, dv, cu_seqlens,
                                  (cudaStream_t)stream);
}

int gla_chunk_bwd_saved(const void *q, const void *k, const void *v, const void *dout, const float *log_decay,
                        const float *h0, const float *dhT, const void *state_images, void *dq, void *dk_out,
                        void *dv_out, float *dh0, int B, int T, int H, int dk, int dv, int chunk,
                        const int32_t *cu_seqlens, void *stream) {
    int rc = check_backward(q, k, v, dout, log_decay, h0, dhT, dq, dk_out, dv_out, dh0, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    if (!state_images) return GLA_ERR_ARG;
    if (!aligned16(state_images)) return GLA_ERR_ALIGN;
    if (!(tc_chunk_len(chunk) && tc_bwd_supported(dk, dv, 128))) return GLA_ERR_UNSUPPORTED;
    return tc_chunk_bwd_bf16_saved(q, k, v, dout, log_decay, h0, dhT, state_images, dq, dk_out, dv_out, dh0, B, T, H,
                                   dk, dv, cu_seqlens, (cudaStream_t)stream);
}

int gla_chunk_bwd_f32(const float *q, const float *k, const float *v, const float *dout, const float *log_decay,
                      const float *h0, const float *dhT, float *dq, float *dk_out, float *dv_out, float *dh0, int B,
                      int T, int H, int dk, int dv, int chunk, const int32_t *cu_seqlens, void *stream) {
    int rc = check_backward(q, k, v, dout, log_decay, h0, dhT, dq, dk_out, dv_out, dh0, B, T, H, dk, dv, cu_seqlens);
    if (rc) return rc;
    return simt_chunk_bwd_f32(q, k, v, dout, log_decay, h0, dhT, dq, dk_out, dv_out, dh0, B, T, H, dk, dv, chunk,
                              cu_seqlens, (cudaStream_t)stream);
}

int gla_decode_step(const void *q, const void *k, const void *v, const float *log_decay, float *state_inout,
                    void *out, int N, int H, int dk, int dv, void *stream) {
    int rc = check_decode(q, k, v, log_decay, state_inout, out, N, H, dk, dv);
    if (rc) return rc;
    return decode_step_bf16(q, k, v, log_decay, state_inout, out, N, H, dk, dv, (cudaStream_t)stream);
}

int gla_decode_step_f32(const float *q, const float *k, const float *v, const float *log_decay,
                        float *state_inout, float *out, int N, int H, int dk, int dv, void *stream) {
    int rc = check_decode(q, k, v, log_decay, state_inout, out, N, H, dk, dv);
    if (rc) return rc;
    return decode_step_f32(q, k, v, log_decay, state_inout, out, N, H, dk, dv, (cudaStream_t)stream);
}

int gla_decode_step_paged(const void *q, const void *k, const void *v, const float *log_decay, float *state_pool,
                          const int32_t *slots, int nslots, void *out, int N, int H, int dk, int dv, void *stream) {
    if (!slots || nslots <= 0) return GLA_ERR_ARG;
    int rc = check_decode(q, k, v, log_decay, state_pool, out, N, H, dk, dv);
    if (rc) return rc;
    if (!aligned16(slots)) return GLA_ERR_ALIGN;
    if ((long long)nslots * H > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    return decode_step_paged_bf16(q, k, v, log_decay, state_pool, slots, nslots, out, N, H, dk, dv,
                                  (cudaStream_t)stream);
}

int gla_decode_step_gated(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                          const float *log_decay, float *state_inout, void *out, int N, int H, int dk, int dv,
                          void *stream) {
    if (!g) return GLA_ERR_ARG;
    if (gate_kind != GLA_GATE_SILU && gate_kind != GLA_GATE_SIGMOID) return GLA_ERR_ARG;
    int rc = check_decode(q, k, v, log_decay, state_inout, out, N, H, dk, dv);
    if (rc) return rc;
    if (!aligned16(g)) return GLA_ERR_ALIGN;
    return decode_step_gated_bf16(q, k, v, g, gate_kind, log_decay, state_inout, nullptr, 0, out, N, H, dk, dv,
                                  (cudaStream_t)stream);
}

int gla_decode_step_paged_gated(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                                const float *log_decay, float *state_pool, const int32_t *slots, int nslots,
                                void *out, int N, int H, int dk, int dv, void *stream) {
    if (!g || !slots || nslots <= 0) return GLA_ERR_ARG;
    if (gate_kind != GLA_GATE_SILU && gate_kind != GLA_GATE_SIGMOID) return GLA_ERR_ARG;
    int rc = check_decode(q, k, v, log_decay, state_pool, out, N, H, dk, dv);
    if (rc) return rc;
    if (!aligned16(g) || !aligned16(slots)) return GLA_ERR_ALIGN;
    if ((long long)nslots * H > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    return decode_step_gated_bf16(q, k, v, g, gate_kind, log_decay, state_pool, slots, nslots, out, N, H, dk, dv,
                                  (cudaStream_t)stream);
}

int gla_decode_step_layers(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                           const float *log_decay, float *state_pool, const int32_t *slots, int nslots,
                           int page_layers, int layer0, int L, void *out, int N, int H, int dk, int dv,
                           void *stream) {
    if (!slots || nslots <= 0 || L <= 0 || page_layers <= 0 || layer0 < 0 || layer0 > page_layers - L)
        return GLA_ERR_ARG;
    if (g && gate_kind != GLA_GATE_SILU && gate_kind != GLA_GATE_SIGMOID) return GLA_ERR_ARG;
    if (N <= 0 || (long long)L * N > 0x7fffffffLL) return GLA_ERR_ARG;
    int rc = check_decode(q, k, v, log_decay, state_pool, out, L * N, H, dk, dv);
    if (rc) return rc;
    if (!aligned16(g) || !aligned16(slots)) return GLA_ERR_ALIGN;
    if ((long long)L * N * H > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    return decode_step_layers_bf16(q, k, v, g, gate_kind, log_decay, state_pool, slots, nslots, page_layers, layer0,
                                   L, out, N, H, dk, dv, (cudaStream_t)stream);
}

int gla_conv1d_silu(const void *x, const float *weight, const float *bias, const float *state_in, float *state_out,
                    void *y, int B, int T, int D, const int32_t *cu_seqlens, void *stream) {
    int rc = check_conv(x, weight, bias, state_in, state_out, y, B, T, D);
    if (rc) return rc;
    if (!aligned16(cu_seqlens)) return GLA_ERR_ALIGN;
    return conv1d_silu_bf16(x, weight, bias, state_in, state_out, y, B, T, D, cu_seqlens, (cudaStream_t)stream);
}

int gla_conv1d_silu_f32(const float *x, const float *weight, const float *bias, const float *state_in,
                        float *state_out, float *y, int B, int T, int D, const int32_t *cu_seqlens, void *stream) {
    int rc = check_conv(x, weight, bias, state_in, state_out, y, B, T, D);
    if (rc) return rc;
    if (!aligned16(cu_seqlens)) return GLA_ERR_ALIGN;
    return conv1d_silu_f32(x, weight, bias, state_in, state_out, y, B, T, D, cu_seqlens, (cudaStream_t)stream);
}

int gla_conv1d_silu_step(const void *x, const float *weight, const float *bias, float *state_inout, void *y, int N,
                         int D, void *stream) {
    if (!state_inout) return GLA_ERR_ARG;
    int rc = check_conv(x, weight, bias, state_inout, state_inout, y, N, 1, D);
    if (rc) return rc;
    return conv1d_silu_step_bf16(x, weight, bias, state_inout, y, N, D, (cudaStream_t)stream);
}

int gla_last_device_status(void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    int result = GLA_OK;
    const int parts[5] = {take_status_simt(st), take_status_decode(st), take_status_tc(st), take_status_bwd(st),
                          take_status_conv(st)};
    for (int p : parts) {
        if (p == GLA_ERR_LAUNCH) return GLA_ERR_LAUNCH;
        if (result == GLA_OK && p != 0) result = p;
    }
    return result;
}

const char *gla_status_str(int status) {
    switch (status) {
        case GLA_OK: return "ok";
        case GLA_ERR_ARG: return "invalid argument";
        case GLA_ERR_UNSUPPORTED: return "unsupported shape, chunk or device";
        case GLA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case GLA_ERR_LAUNCH: return "CUDA call or kernel launch failed";
        case GLA_ERR_TIMEOUT: return "device pipeline wait timed out";
        case GLA_ERR_NOMEM: return "scratch allocation failed";
        case GLA_ERR_DEVICE_ARG: return "invalid cu_seqlens found on the device";
        case GLA_ERR_SCRATCH_LIMIT: return "problem needs more segment-state scratch than the fixed no-alloc array";
        default: return "unknown status";
    }
}

int gla_chunk_kernel(int op, int dtype, int dk, int dv, int chunk) {
    if (op != GLA_OP_FORWARD && op != GLA_OP_FORWARD_GATED && op != GLA_OP_BACKWARD) return GLA_ERR_ARG;
    if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_ARG;
    if (dk < 16 || dk > 256 || dv < 16 || dv > 512 || dk % 8 || dv % 8) return GLA_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return GLA_ERR_UNSUPPORTED;
    if (!device_info().ok) return GLA_ERR_UNSUPPORTED;
    if (dtype == GLA_F32 || !tc_chunk_len(chunk)) return GLA_KERNEL_SIMT;
    const bool tc = op == GLA_OP_FORWARD         ? tc_chunk_supported(dk, dv, 128)
                    : op == GLA_OP_FORWARD_GATED ? tc_gate_supported(dk, dv)
                                                 : tc_bwd_supported(dk, dv, 128);
    return tc ? GLA_KERNEL_TENSOR_CORE : GLA_KERNEL_SIMT;
}

uint64_t gla_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int gla_version(void) { return 200; }

}  // extern "C"
