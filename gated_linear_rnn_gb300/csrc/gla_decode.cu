// gla_decode.cu — one recurrent Simple GLA decode step (memory-bound).
//
// Page "线性注意力模型如何实现固定推理状态", section "i14 与 Laplace 3B 架构":
// inference costs O(1) per token because the dk x dv state per head has a fixed
// size; section "Trainium2 上的推理优化": each sequence owns one fixed state page.
// For every (sequence n, head h):
//     S <- lambda_h S + k^T v      (in place)
//     o  = q S                     (updated S)
//
// The step is bound by HBM: every state element is read once and written once
// (8 bytes per element, 147,456 bytes for a 96 x 192 head) against 2 FLOP of
// update and 2 FLOP of read-out.  One CTA owns one (n, h) state tile.  Its
// threads form RG row groups x (dv/4) column groups; each thread streams rows
// rg, rg+RG, ... of its 4-column slice with 16-byte loads and stores (a warp
// covers 512 contiguous bytes of a row), issuing UNROLL loads before using any
// of them so that enough bytes are in flight per SM.  The read-out sum over dk
// is finished through shared memory across the row groups.
//
// Paged form (same section: the serving engine gives every sequence one fixed
// state page in its pool, and every new batch width was a separate compiled
// shape, so batches were padded to a fixed width): the state of batch row n is
// page slots[n] of a pool of nslots pages; a negative slot marks a padding row,
// whose output is zero and which touches no page.  The kernel is the same for
// every width, and a fixed-width padded call can be captured in a CUDA graph
// and replayed with new slot tables.
#include "gla_common.cuh"

GLA_DEFINE_STATUS(decode)

namespace gla {
namespace {

constexpr int kRG = 4;  // row groups per CTA

template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&x)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&x)[4]) {
    const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&x)[4]) {
    const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&t.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&t.y);
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
}

// kMaxThreads bounds the block (and so the register budget); kUnroll state rows are in flight per
// thread: 12 for blocks of up to 256 threads (dv <= 256), 4 for the wide blocks.
template <typename T, int kMaxThreads, int kUnroll>
__global__ void __launch_bounds__(kMaxThreads)
decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const float *__restrict__ log_decay, float *__restrict__ state, T *__restrict__ out,
              int H, int dk, int dv, const int32_t *__restrict__ slots, int nslots, const T *__restrict__ gate,
              int gate_kind, int rows, int page_layers, int layer0) {
    extern __shared__ float sm[];
    float *qs = sm, *ks = sm + dk, *red = sm + 2 * dk;  // red: [kRG][dv]
    // unit = (l * rows + n) * H + h: layer l of the call, batch row n, head h (one layer: l = 0)
    const int unit = blockIdx.x;
    const int h = unit % H;
    const int n = (unit / H) % rows, l = unit / (H * rows);
    const int ncg = dv >> 2;
    const int tid = threadIdx.x;
    const int cg = tid % ncg, rg = tid / ncg;
    // the slot (paged form) and q, k, v are independent loads: all in flight at once
    const int slot = slots != nullptr ? __ldg(slots + n) : 0;
    for (int i = tid; i < dk; i += blockDim.x) {
        qs[i] = to_f32(q[(size_t)unit * dk + i]);
        ks[i] = to_f32(k[(size_t)unit * dk + i]);
    }
    float vv[4];
    load4<T>(v + (size_t)unit * dv + cg * 4, vv);
    const float lam = expf(__ldg(log_decay + (size_t)l * H + h));
    size_t page = (size_t)unit;  // state page of this (n, h): unit itself unless paged
    if (slots != nullptr) {
        if (slot < 0 || slot >= nslots) {  // padding row (or a bad slot, reported): zero output, no page
            if (slot >= nslots && tid == 0) record_status(GLA_ERR_DEVICE_ARG);
            for (int c = tid; c < dv; c += blockDim.x) out[(size_t)unit * dv + c] = from_f32<T>(0.f);
            return;
        }
        page = ((size_t)slot * page_layers + layer0 + l) * H + h;  // layer layer0 + l of page `slot`
    }

    float4 *S = reinterpret_cast<float4 *>(state + page * dk * dv) + cg;
    const int row_f4 = ncg;  // float4 per state row
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float4 s[kUnroll];
    // the first rows of state need neither q nor k: in flight before the block barrier
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int r = rg + u * kRG;
        if (r < dk) s[u] = __ldcs(S + (size_t)r * row_f4);
    }
    __syncthreads();
    for (int r0 = rg; r0 < dk; r0 += kRG * kUnroll) {
        if (r0 != rg) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int r = r0 + u * kRG;
                if (r < dk) s[u] = __ldcs(S + (size_t)r * row_f4);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int r = r0 + u * kRG;
            if (r < dk) {
                const float kr = ks[r], qr = qs[r];
                float4 t = s[u];
                t.x = fmaf(lam, t.x, kr * vv[0]);
                t.y = fmaf(lam, t.y, kr * vv[1]);
                t.z = fmaf(lam, t.z, kr * vv[2]);
                t.w = fmaf(lam, t.w, kr * vv[3]);
                acc[0] = fmaf(qr, t.x, acc[0]);
                acc[1] = fmaf(qr, t.y, acc[1]);
                acc[2] = fmaf(qr, t.z, acc[2]);
                acc[3] = fmaf(qr, t.w, acc[3]);
                __stcs(S + (size_t)r * row_f4, t);
            }
        }
    }
    *reinterpret_cast<float4 *>(red + rg * dv + cg * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncthreads();
    for (int c = tid; c < dv; c += blockDim.x) {
        float o = 0.f;
#pragma unroll
        for (int g = 0; g < kRG; ++g) o += red[g * dv + c];
        if (gate != nullptr) o *= gate_factor(to_f32(gate[(size_t)unit * dv + c]), gate_kind);
        out[(size_t)unit * dv + c] = from_f32<T>(o);
    }
}

template <typename T>
int launch_decode(const T *q, const T *k, const T *v, const float *ld, float *state, T *out, int N, int H,
                  int dk, int dv, cudaStream_t st, const int32_t *slots = nullptr, int nslots = 0,
                  const T *gate = nullptr, int gate_kind = 0, int L = 1, int page_layers = 1, int layer0 = 0) {
    const long long units = (long long)L * N * H;
    if (units > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    const int threads = (dv / 4) * kRG;
    if (threads > 1024) return GLA_ERR_UNSUPPORTED;
    const size_t bytes = (size_t)(2 * dk + kRG * dv) * sizeof(float);
    if (threads <= 256)
        decode_kernel<T, 256, 12><<<(unsigned)units, threads, bytes, st>>>(q, k, v, ld, state, out, H, dk, dv,
                                                                           slots, nslots, gate, gate_kind, N,
                                                                           page_layers, layer0);
    else
        decode_kernel<T, 1024, 4><<<(unsigned)units, threads, bytes, st>>>(q, k, v, ld, state, out, H, dk, dv,
                                                                           slots, nslots, gate, gate_kind, N,
                                                                           page_layers, layer0);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

}  // namespace

int decode_step_bf16(const void *q, const void *k, const void *v, const float *ld, float *state, void *out,
                     int N, int H, int dk, int dv, cudaStream_t st) {
    using B = __nv_bfloat16;
    return launch_decode<B>((const B *)q, (const B *)k, (const B *)v, ld, state, (B *)out, N, H, dk, dv, st);
}

int decode_step_f32(const float *q, const float *k, const float *v, const float *ld, float *state, float *out,
                    int N, int H, int dk, int dv, cudaStream_t st) {
    return launch_decode<float>(q, k, v, ld, state, out, N, H, dk, dv, st);
}

int decode_step_paged_bf16(const void *q, const void *k, const void *v, const float *ld, float *pool,
                           const int32_t *slots, int nslots, void *out, int N, int H, int dk, int dv,
                           cudaStream_t st) {
    using B = __nv_bfloat16;
    return launch_decode<B>((const B *)q, (const B *)k, (const B *)v, ld, pool, (B *)out, N, H, dk, dv, st, slots,
                            nslots);
}

// L layers of a step in one launch: q, k [L, N, H, dk], v, out (and gate) [L, N, H, dv], log_decay
// [L, H]; layer l of row n uses layer layer0 + l of page slots[n] in a pool of pages of page_layers
// layers ([nslots, page_layers, H, dk, dv]).
int decode_step_layers_bf16(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                            const float *ld, float *pool, const int32_t *slots, int nslots, int page_layers,
                            int layer0, int L, void *out, int N, int H, int dk, int dv, cudaStream_t st) {
    using B = __nv_bfloat16;
    return launch_decode<B>((const B *)q, (const B *)k, (const B *)v, ld, pool, (B *)out, N, H, dk, dv, st, slots,
                            nslots, (const B *)g, gate_kind, L, page_layers, layer0);
}

// The step with the output gate applied to o (slots null: the dense state layout).
int decode_step_gated_bf16(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                           const float *ld, float *state, const int32_t *slots, int nslots, void *out, int N, int H,
                           int dk, int dv, cudaStream_t st) {
    using B = __nv_bfloat16;
    return launch_decode<B>((const B *)q, (const B *)k, (const B *)v, ld, state, (B *)out, N, H, dk, dv, st, slots,
                            nslots, (const B *)g, gate_kind);
}

}  // namespace gla
