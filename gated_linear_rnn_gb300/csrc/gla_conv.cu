// gla_conv.cu — causal depthwise Conv1d of width 4 + SiLU (memory-bound).
//
// Page "线性注意力模型如何实现固定推理状态", section "i14 与 Laplace 3B 架构"
// ("归一化与卷积"): every position of the normalised residual stream gets a
// 4-token summary from a per-channel causal Conv1d of width k = 4 with SiLU,
// before the QKVG projection.  For channel c at token t of a sequence:
//     z = b[c] + sum_{k=0..3} w[c][k] x_{t-3+k}[c]     (w[c][3] meets x_t)
//     y = z * sigmoid(z)
// The three inputs before a sequence's first token come from its conv state
// (oldest first; zeros without one), and the state after it holds its last
// three inputs, so a sequence can be continued in a later call or by the
// per-token step below.
//
// Prefill: a thread owns 8 consecutive channels (one 16-byte bf16 vector) and
// a run of 8 rows, all loaded at once, with the three inputs before its current
// row in registers; a warp covers 256 channels = 512 contiguous bytes of a row.
// The three rows before a run are read again by it (through L2), so HBM sees
// every input about once and every output once (4 bytes per element for
// bf16).  Step: one thread per 8 channels of one sequence.
#include "gla_common.cuh"

GLA_DEFINE_STATUS(conv)

namespace gla {
namespace {

constexpr int kThreads = 256;  // prefill: 8 runs x 256 channels per block; step: 2048 channels
constexpr int kVec = 8;        // channels per thread
constexpr int kRun = 8;        // rows per thread in the prefill kernel, all loaded before the first is used

template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
    typedef uint4 Raw;
    // inputs are read through the cached path: the three rows before a run are read again by it
    static __device__ __forceinline__ Raw load_raw(const __nv_bfloat16 *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
    static __device__ __forceinline__ void unpack(const Raw &u, float (&x)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&x)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&y)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&b);
        }
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
    }
};
template <>
struct Vec8<float> {
    struct Raw {
        float4 a, b;
    };
    static __device__ __forceinline__ Raw load_raw(const float *p) {
        return Raw{__ldg(reinterpret_cast<const float4 *>(p)), __ldg(reinterpret_cast<const float4 *>(p) + 1)};
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[8]) {
        x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w; x[4] = r.b.x; x[5] = r.b.y; x[6] = r.b.z; x[7] = r.b.w;
    }
    static __device__ __forceinline__ void load(const float *p, float (&x)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&y)[8]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(y[0], y[1], y[2], y[3]));
        __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(y[4], y[5], y[6], y[7]));
    }
};

// SiLU with the fast exponential and division intrinsics: the kernel is bound by instruction issue
// long before HBM with the IEEE forms (about 40 instructions per element).  z is clamped at -80
// so that 1 + e^-z stays finite (the result there is below 2e-33 in magnitude either way).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-fmaxf(z, -80.f))); }

// For bf16 outputs: sigmoid(z) = (1 + tanh(z/2)) / 2 with the hardware tanh approximation
// (relative error about 2^-11, well inside the bf16 rounding of the result): three instructions.
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
template <typename T>
__device__ __forceinline__ float silu_t(float z) { return silu(z); }
template <>
__device__ __forceinline__ float silu_t<__nv_bfloat16>(float z) {
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_approx(hz), hz);
}

// sequence of `row` and its [start, end) rows; dense batches have cu == null
__device__ __forceinline__ int seq_of(int64_t row, int nseq, int T, const int32_t *cu, int64_t &start,
                                      int64_t &end) {
    if (cu == nullptr) {
        const int s = (int)(row / T);
        start = (int64_t)s * T;
        end = start + T;
        return s;
    }
    int lo = 0, hi = nseq - 1;  // last s with cu[s] <= row and cu[s + 1] > row
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= row) lo = mid;
        else hi = mid - 1;
    }
    int s = lo;
    while (s < nseq - 1 && __ldg(cu + s + 1) <= row) ++s;  // skip empty sequences
    start = __ldg(cu + s);
    end = __ldg(cu + s + 1);
    return s;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
conv_prefill_kernel(const T *__restrict__ x, const float *__restrict__ w, const float *__restrict__ b,
                    const float *__restrict__ st_in, float *__restrict__ st_out, T *__restrict__ y, int64_t rows,
                    int nseq, int Tlen, int D, const int32_t *__restrict__ cu) {
    // a warp covers 256 channels (512 contiguous bytes per row) of a run of kRun rows; a thread keeps
    // the three inputs before its current row in registers and loads its whole run at once
    const int c0 = (blockIdx.y * 32 + (threadIdx.x & 31)) * kVec;
    const int64_t r0 = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kRun;
    if (c0 >= D || r0 >= rows) return;
    const int64_t valid_rows = cu ? (int64_t)__ldg(cu + nseq) : rows;  // rows past the last sequence: untouched
    if (r0 >= valid_rows) return;
    const int64_t r1 = (r0 + kRun < valid_rows) ? r0 + kRun : valid_rows;
    typename Vec8<T>::Raw xr[kRun];
#pragma unroll
    for (int j = 0; j < kRun; ++j)
        if (r0 + j < r1) xr[j] = Vec8<T>::load_raw(x + (size_t)(r0 + j) * D + c0);
    int64_t start, end;
    int s = seq_of(r0, nseq, Tlen, cu, start, end);
    if (start < 0 || start > r0 || end <= r0 || end > rows) {
        record_status(GLA_ERR_DEVICE_ARG);
        return;
    }
    float h[3][8];  // x_{t-3}, x_{t-2}, x_{t-1}
    auto fill_history = [&](int64_t row) {
        for (int m = 0; m < 3; ++m) {
            const int64_t q = row - 3 + m;  // absolute row of that input
            if (q >= start) {
                Vec8<T>::unpack(Vec8<T>::load_raw(x + (size_t)q * D + c0), h[m]);
            } else {
                const int idx = (int)(q - start) + 3;  // 0..2 within the incoming state
#pragma unroll
                for (int i = 0; i < kVec; ++i)
                    h[m][i] = st_in ? __ldg(st_in + ((size_t)s * D + c0 + i) * 3 + idx) : 0.f;
            }
        }
    };
    fill_history(r0);
    float wt[4][8], bias[8];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(w + (size_t)(c0 + i) * 4));
        wt[0][i] = t.x; wt[1][i] = t.y; wt[2][i] = t.z; wt[3][i] = t.w;
        bias[i] = b ? __ldg(b + c0 + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kRun; ++j) {
        const int64_t row = r0 + j;
        if (row >= r1) break;
        if (row >= end) {  // the next sequence starts inside this run
            s = seq_of(row, nseq, Tlen, cu, start, end);
            if (start < 0 || start > row || end <= row || end > rows) {
                record_status(GLA_ERR_DEVICE_ARG);
                return;
            }
            fill_history(row);
        }
        float xt[8], out[8];
        Vec8<T>::unpack(xr[j], xt);
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            const float z = bias[i] + wt[0][i] * h[0][i] + wt[1][i] * h[1][i] + wt[2][i] * h[2][i] + wt[3][i] * xt[i];
            out[i] = silu_t<T>(z);
            h[0][i] = h[1][i];
            h[1][i] = h[2][i];
            h[2][i] = xt[i];
        }
        Vec8<T>::store(y + (size_t)row * D + c0, out);
        if (row == end - 1 && st_out) {  // last token of the sequence: its conv state
#pragma unroll
            for (int i = 0; i < kVec; ++i)
#pragma unroll
                for (int m = 0; m < 3; ++m) st_out[((size_t)s * D + c0 + i) * 3 + m] = h[m][i];
        }
    }
}

// Sequences without tokens pass their conv state through (zeros without one).
__global__ void conv_empty_kernel(const float *__restrict__ st_in, float *__restrict__ st_out, int nseq, int D,
                                  const int32_t *__restrict__ cu) {
    const int s = blockIdx.x;
    if (__ldg(cu + s + 1) != __ldg(cu + s)) return;
    for (int e = threadIdx.x; e < D * 3; e += blockDim.x)
        st_out[(size_t)s * D * 3 + e] = st_in ? st_in[(size_t)s * D * 3 + e] : 0.f;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
conv_step_kernel(const T *__restrict__ x, const float *__restrict__ w, const float *__restrict__ b,
                 float *__restrict__ state, T *__restrict__ y, int N, int D) {
    const int c0 = (blockIdx.x * kThreads + threadIdx.x) * kVec;
    const int n = blockIdx.y;
    if (c0 >= D || n >= N) return;
    float xt[8], out[8];
    Vec8<T>::load(x + (size_t)n * D + c0, xt);
    float4 *sp = reinterpret_cast<float4 *>(state + ((size_t)n * D + c0) * 3);  // 24 floats, 16-byte aligned
    float hs[24];
#pragma unroll
    for (int j = 0; j < 6; ++j) {
        const float4 t = sp[j];
        hs[4 * j] = t.x; hs[4 * j + 1] = t.y; hs[4 * j + 2] = t.z; hs[4 * j + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(w + (size_t)(c0 + i) * 4));
        const float z = (b ? __ldg(b + c0 + i) : 0.f) + t.x * hs[3 * i] + t.y * hs[3 * i + 1] + t.z * hs[3 * i + 2] +
                        t.w * xt[i];
        out[i] = silu(z);
        hs[3 * i] = hs[3 * i + 1];
        hs[3 * i + 1] = hs[3 * i + 2];
        hs[3 * i + 2] = xt[i];
    }
#pragma unroll
    for (int j = 0; j < 6; ++j) sp[j] = make_float4(hs[4 * j], hs[4 * j + 1], hs[4 * j + 2], hs[4 * j + 3]);
    Vec8<T>::store(y + (size_t)n * D + c0, out);
}

}  // namespace

template <typename T>
static int conv_prefill(const T *x, const float *w, const float *b, const float *st_in, float *st_out, T *y, int nseq,
                        int Tlen, int D, const int32_t *cu, cudaStream_t st) {
    const int64_t rows = cu ? (int64_t)Tlen : (int64_t)nseq * Tlen;
    const int64_t tiles = (rows + kRun * (kThreads / 32) - 1) / (kRun * (kThreads / 32));
    const int cgroups = (D / kVec + 31) / 32;
    if (tiles > 0x7fffffffLL || cgroups > 65535) return GLA_ERR_UNSUPPORTED;
    if (rows > 0) {
        dim3 grid((unsigned)tiles, (unsigned)cgroups);
        conv_prefill_kernel<T><<<grid, kThreads, 0, st>>>(x, w, b, st_in, st_out, y, rows, nseq, Tlen, D, cu);
        count_launches(1);
    }
    if (cu != nullptr && st_out != nullptr && nseq > 0) {
        conv_empty_kernel<<<nseq, 256, 0, st>>>(st_in, st_out, nseq, D, cu);
        count_launches(1);
    }
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

int conv1d_silu_bf16(const void *x, const float *w, const float *b, const float *st_in, float *st_out, void *y,
                     int nseq, int Tlen, int D, const int32_t *cu, cudaStream_t st) {
    using B = __nv_bfloat16;
    return conv_prefill<B>((const B *)x, w, b, st_in, st_out, (B *)y, nseq, Tlen, D, cu, st);
}

int conv1d_silu_f32(const float *x, const float *w, const float *b, const float *st_in, float *st_out, float *y,
                    int nseq, int Tlen, int D, const int32_t *cu, cudaStream_t st) {
    return conv_prefill<float>(x, w, b, st_in, st_out, y, nseq, Tlen, D, cu, st);
}

int conv1d_silu_step_bf16(const void *x, const float *w, const float *b, float *state, void *y, int N, int D,
                          cudaStream_t st) {
    using B = __nv_bfloat16;
    const int cgroups = (D / kVec + kThreads - 1) / kThreads;
    if (N > 65535) return GLA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)cgroups, (unsigned)N);
    conv_step_kernel<B><<<grid, kThreads, 0, st>>>((const B *)x, w, b, state, (B *)y, N, D);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

}  // namespace gla
