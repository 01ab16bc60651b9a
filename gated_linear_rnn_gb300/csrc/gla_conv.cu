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
// Prefill: a TMA pipeline over 64-row tiles of a 256-channel slab (the box also
// carries the three rows before the tile), a lane owning 8 channels of 8 rows
// with the three inputs before its row in registers (details at the kernel).
// HBM sees every input about once (the three extra rows per tile come from L2)
// and every output once.  Step: one thread per 8 channels of one sequence.
#include <cuda.h>

#include <atomic>

#include "gla_common.cuh"
#include "sm100_ptx.cuh"

GLA_DEFINE_STATUS(conv)

namespace gla {
namespace {

constexpr int kVec = 8;        // channels per thread

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
// SiLU of the prefill kernel, whose argument comes scaled: z itself for f32, z / 2 for bf16 (the tanh form)
template <typename T>
__device__ __forceinline__ float silu_scaled(float z) { return silu(z); }
template <>
__device__ __forceinline__ float silu_scaled<__nv_bfloat16>(float hz) { return fmaf(hz, tanh_approx(hz), hz); }

// Two f32 lanes per instruction: fma.rn.f32x2 rounds each lane as fma.rn.f32 does, so the paired
// arithmetic below gives the scalar form's results bit for bit with half the FMA instructions.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// a bf16 pair (channels 2i, 2i+1 of one row) as an f32 pair
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
    return ((uint64_t)(w & 0xffff0000u) << 32) | (uint64_t)(w << 16);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
// One output row of a lane's 8 bf16 channels: z/2 = b/2 + sum_k (w_k/2) x_k in the order of the scalar
// form, then hz + hz tanh(hz), as f32 pairs; x_k are the lane's 16 bytes of input rows t-3+k.
__device__ __forceinline__ uint4 conv_row_bf16(const uint64_t (&w2)[4][4], const uint64_t (&b2)[4], const uint4 &x0,
                                               const uint4 &x1, const uint4 &x2, const uint4 &x3) {
    const uint32_t a0[4] = {x0.x, x0.y, x0.z, x0.w}, a1[4] = {x1.x, x1.y, x1.z, x1.w};
    const uint32_t a2[4] = {x2.x, x2.y, x2.z, x2.w}, a3[4] = {x3.x, x3.y, x3.z, x3.w};
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint64_t z = fma_f32x2(w2[0][p], bf16x2_to_f32x2(a0[p]), b2[p]);
        z = fma_f32x2(w2[1][p], bf16x2_to_f32x2(a1[p]), z);
        z = fma_f32x2(w2[2][p], bf16x2_to_f32x2(a2[p]), z);
        z = fma_f32x2(w2[3][p], bf16x2_to_f32x2(a3[p]), z);
        float zl, zh;
        f32x2_split(z, zl, zh);
        const uint64_t y = fma_f32x2(z, f32x2(tanh_approx(zl), tanh_approx(zh)), z);
        float yl, yh;
        f32x2_split(y, yl, yh);
        o[p] = pack_bf16x2(yl, yh);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
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

// Prefill pipeline.  A CTA owns a slab of up to 256 channels and walks 64-row tiles of it (tile t,
// then t + gridDim.x, ...).  A producer warp brings each tile in with one TMA box that also holds the
// three rows before the tile (rows from -3 are zero-filled), into a ring of shared-memory stages; eight
// compute warps take 8 rows each: a lane owns 8 channels, keeps the three inputs before its row in
// registers and stores its 16 bytes of y, so a warp writes whole 512-byte rows.  The bytes in flight
// are the stages in shared memory, not registers.
constexpr int kCvWarps = 8;                     // compute warps
constexpr int kCvRun = 8;                       // rows per compute warp and tile
constexpr int kCvTile = kCvWarps * kCvRun;      // 64 rows per tile
constexpr int kCvBoxRows = kCvTile + 3;         // + the three rows before the tile
constexpr int kCvThreads = (kCvWarps + 1) * 32; // + the producer warp
constexpr int kCvSlab = 256;                    // channels per CTA (the TMA box is at most 256 wide)
constexpr uint64_t kCvWaitNs = 2000000000ull;   // 2 s per wait

template <typename T> struct CvStages;
template <> struct CvStages<__nv_bfloat16> { static constexpr int n = 3; };  // 3 x 33.5 KB
template <> struct CvStages<float> { static constexpr int n = 2; };          // 2 x 67 KB

// 8 channels of one staged row (the lane's 16 bytes of bf16, or 32 bytes of f32)
__device__ __forceinline__ void row8(const uint8_t *row, int lane, float (&x)[8], const __nv_bfloat16 *) {
    Vec8<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(row + 16 * lane), x);
}
__device__ __forceinline__ void row8(const uint8_t *row, int lane, float (&x)[8], const float *) {
    const float4 a = *reinterpret_cast<const float4 *>(row + 32 * lane);
    const float4 b = *reinterpret_cast<const float4 *>(row + 32 * lane + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// 104 registers and no spills (a launch bound for two CTAs per SM makes the compiler stop at 96 and spill
// inside the row loop).  One CTA then fits per SM: each of the SM's four sub-partitions holds 16 K
// registers, and two CTAs of nine warps would put five warps on one of them.
template <typename T>
__global__ void __maxnreg__(104)
conv_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const float *__restrict__ w, const float *__restrict__ b,
                    const float *__restrict__ st_in, float *__restrict__ st_out, T *__restrict__ y, int64_t rows,
                    int nseq, int Tlen, int D, int slab, const int32_t *__restrict__ cu, int64_t ntiles) {
    using namespace ptx;
    constexpr int NST = CvStages<T>::n;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t row_bytes = (uint32_t)slab * sizeof(T);
    const uint32_t stage_bytes = (uint32_t)kCvBoxRows * row_bytes;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + NST * stage_bytes;  // 8-byte aligned: row_bytes is a multiple of 16
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + NST * stage_bytes + 16 * NST);
    auto full = [&](int st) { return bar0 + 8u * (uint32_t)st; };
    auto empty = [&](int st) { return bar0 + 8u * (uint32_t)(NST + st); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cbase = blockIdx.y * slab;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int st = 0; st < NST; ++st) {
            mbar_init(full(st), 1);
            mbar_init(empty(st), kCvWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCvWarps) {
        // ---- producer: one TMA box per tile, box row k = row t * 64 - 3 + k ----
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            int64_t i = 0;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int st = (int)(i % NST);
                if (i >= NST && !mbar_wait(empty(st), (uint32_t)((i / NST) - 1) & 1u, abort_flag, kCvWaitNs)) {
                    record_status(GLA_ERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                mbar_expect_tx(full(st), stage_bytes);
                tma_load_2d(sbase + (uint32_t)st * stage_bytes, &tmX, cbase, (int32_t)(t * kCvTile - 3), full(st));
            }
        }
        return;
    }

    // ---- compute warps ----
    const int c0 = cbase + 8 * lane;
    const bool active = 8 * lane < slab && c0 < D;
    const int64_t valid_rows = cu ? (int64_t)__ldg(cu + nseq) : rows;  // rows past the last sequence: untouched
    // for bf16 outputs SiLU is computed as hz + hz tanh(hz) with hz = z / 2, so the fast path carries the
    // weights and bias halved (exact: a power of two)
    constexpr float kZs = sizeof(T) == 2 ? 0.5f : 1.f;
    float wt[4][8], bias[8];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
        const float4 t4 = active ? __ldg(reinterpret_cast<const float4 *>(w + (size_t)(c0 + i) * 4))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        wt[0][i] = kZs * t4.x; wt[1][i] = kZs * t4.y; wt[2][i] = kZs * t4.z; wt[3][i] = kZs * t4.w;
        bias[i] = (active && b) ? kZs * __ldg(b + c0 + i) : 0.f;
    }
    int64_t i = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
        const int st = (int)(i % NST);
        if (!mbar_wait(full(st), (uint32_t)(i / NST) & 1u, abort_flag, kCvWaitNs)) {
            record_status(GLA_ERR_TIMEOUT);
            *abort_flag = 1;
            return;
        }
        const uint8_t *box = smem + (size_t)st * stage_bytes;  // box row k holds row t * 64 - 3 + k
        const uint8_t *wbox = box + (size_t)warp * kCvRun * row_bytes;  // this warp's rows start at box row 3
        const int64_t r0 = t * kCvTile + (int64_t)warp * kCvRun;
        const int64_t r1 = (r0 + kCvRun < valid_rows) ? r0 + kCvRun : valid_rows;
        bool bad = false;
        if (active && r0 < r1) {
            int64_t start, end;
            int s = seq_of(r0, nseq, Tlen, cu, start, end);
            bad = start < 0 || start > r0 || end <= r0 || end > rows;
            if (!bad && r1 == r0 + kCvRun && start <= r0 - 3 && end >= r0 + kCvRun) {
                // fast path: the run and its three inputs before lie inside one sequence; fully unrolled,
                // so the window of the last four rows lives in registers without copies
                T *yp = y + (size_t)r0 * D + c0;
                if constexpr (sizeof(T) == 2) {
                    uint64_t w2[4][4], b2[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) w2[k][p] = f32x2(wt[k][2 * p], wt[k][2 * p + 1]);
                        b2[p] = f32x2(bias[2 * p], bias[2 * p + 1]);
                    }
                    uint4 xr[kCvRun + 3];  // the lane's 16 bytes of each staged row
#pragma unroll
                    for (int m = 0; m < 3; ++m) xr[m] = *reinterpret_cast<const uint4 *>(wbox + (size_t)m * row_bytes + 16 * lane);
#pragma unroll
                    for (int j = 0; j < kCvRun; ++j) {
                        xr[j + 3] = *reinterpret_cast<const uint4 *>(wbox + (size_t)(j + 3) * row_bytes + 16 * lane);
                        __stcs(reinterpret_cast<uint4 *>(yp + (size_t)j * D),
                               conv_row_bf16(w2, b2, xr[j], xr[j + 1], xr[j + 2], xr[j + 3]));
                    }
                    if (end == r0 + kCvRun && st_out) {  // the run ends its sequence: the conv state
#pragma unroll
                        for (int m = 0; m < 3; ++m) {
                            float xm[8];
                            Vec8<__nv_bfloat16>::unpack(xr[kCvRun + m], xm);
#pragma unroll
                            for (int e = 0; e < kVec; ++e) st_out[((size_t)s * D + c0 + e) * 3 + m] = xm[e];
                        }
                    }
                } else {
                    float xw[kCvRun + 3][8];
#pragma unroll
                    for (int m = 0; m < 3; ++m) row8(wbox + (size_t)m * row_bytes, lane, xw[m], (const T *)nullptr);
#pragma unroll
                    for (int j = 0; j < kCvRun; ++j) {
                        row8(wbox + (size_t)(j + 3) * row_bytes, lane, xw[j + 3], (const T *)nullptr);
                        float out[8];
#pragma unroll
                        for (int e = 0; e < kVec; ++e) {
                            const float z = fmaf(wt[3][e], xw[j + 3][e],
                                                 fmaf(wt[2][e], xw[j + 2][e], fmaf(wt[1][e], xw[j + 1][e], fmaf(wt[0][e], xw[j][e], bias[e]))));
                            out[e] = silu_scaled<T>(z);
                        }
                        Vec8<T>::store(yp + (size_t)j * D, out);
                    }
                    if (end == r0 + kCvRun && st_out) {  // the run ends its sequence: the conv state
#pragma unroll
                        for (int e = 0; e < kVec; ++e)
#pragma unroll
                            for (int m = 0; m < 3; ++m) st_out[((size_t)s * D + c0 + e) * 3 + m] = xw[kCvRun + m][e];
                    }
                }
            } else if (!bad) {
                float h[3][8];  // x_{t-3}, x_{t-2}, x_{t-1}
                // inputs before `row`: staged rows, or the incoming conv state before the sequence start
                auto fill_history = [&](int64_t row) {
                    for (int m = 0; m < 3; ++m) {
                        const int64_t q = row - 3 + m;
                        if (q >= start) {
                            row8(box + (size_t)(q - (t * kCvTile - 3)) * row_bytes, lane, h[m], (const T *)nullptr);
                        } else {
                            const int idx = (int)(q - start) + 3;  // 0..2 within the incoming state
#pragma unroll
                            for (int e = 0; e < kVec; ++e)
                                h[m][e] = st_in ? __ldg(st_in + ((size_t)s * D + c0 + e) * 3 + idx) : 0.f;
                        }
                    }
                };
                fill_history(r0);
                for (int j = 0; j < kCvRun; ++j) {
                    const int64_t row = r0 + j;
                    if (row >= r1) break;
                    if (row >= end) {  // the next sequence starts inside this run
                        s = seq_of(row, nseq, Tlen, cu, start, end);
                        if (start < 0 || start > row || end <= row || end > rows) {
                            bad = true;
                            break;
                        }
                        fill_history(row);
                    }
                    float xt[8], out[8];
                    row8(wbox + (size_t)(3 + j) * row_bytes, lane, xt, (const T *)nullptr);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) {
                        const float z = fmaf(wt[3][e], xt[e], fmaf(wt[2][e], h[2][e], fmaf(wt[1][e], h[1][e], fmaf(wt[0][e], h[0][e], bias[e]))));
                        out[e] = silu_scaled<T>(z);
                        h[0][e] = h[1][e];
                        h[1][e] = h[2][e];
                        h[2][e] = xt[e];
                    }
                    Vec8<T>::store(y + (size_t)row * D + c0, out);
                    if (row == end - 1 && st_out) {  // last token of the sequence: its conv state
#pragma unroll
                        for (int e = 0; e < kVec; ++e)
#pragma unroll
                            for (int m = 0; m < 3; ++m) st_out[((size_t)s * D + c0 + e) * 3 + m] = h[m][e];
                    }
                }
            }
        }
        if (bad) record_status(GLA_ERR_DEVICE_ARG);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(st));  // this warp is done with the stage
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

// Step: a block owns 1024 channels (8 per thread) of spb consecutive sequences, so the weights and bias
// are read once per block and reused; two sequences' x and state are in flight at a time.  The host
// picks spb so that the grid is one wave (1280 sequences x 3072 channels: 9 a block, 429 blocks).
constexpr int kStepThreads = 128;
constexpr int kStepSeqs = 8;  // sequences per block when the occupancy cannot be looked up

template <typename T>
__global__ void __launch_bounds__(kStepThreads)
conv_step_kernel(const T *__restrict__ x, const float *__restrict__ w, const float *__restrict__ b,
                 float *__restrict__ state, T *__restrict__ y, int N, int D, int spb) {
    const int c0 = (blockIdx.x * kStepThreads + threadIdx.x) * kVec;
    if (c0 >= D) return;
    const int n0 = blockIdx.y * spb, n1 = min(n0 + spb, N);
    float wt[4][8], bias[8];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(w + (size_t)(c0 + i) * 4));
        wt[0][i] = t.x; wt[1][i] = t.y; wt[2][i] = t.z; wt[3][i] = t.w;
        bias[i] = b ? __ldg(b + c0 + i) : 0.f;
    }
#pragma unroll 1
    for (int nn = n0; nn < n1; nn += 2) {
        float xt[2][8], hs[2][24];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int n = nn + u;
            if (n >= n1) continue;
            Vec8<T>::load(x + (size_t)n * D + c0, xt[u]);
            const float4 *sp = reinterpret_cast<const float4 *>(state + ((size_t)n * D + c0) * 3);  // 24 floats
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                const float4 t = sp[j];
                hs[u][4 * j] = t.x; hs[u][4 * j + 1] = t.y; hs[u][4 * j + 2] = t.z; hs[u][4 * j + 3] = t.w;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int n = nn + u;
            if (n >= n1) continue;
            float out[8];
#pragma unroll
            for (int i = 0; i < kVec; ++i) {
                const float z = bias[i] + wt[0][i] * hs[u][3 * i] + wt[1][i] * hs[u][3 * i + 1] +
                                wt[2][i] * hs[u][3 * i + 2] + wt[3][i] * xt[u][i];
                out[i] = silu(z);
                hs[u][3 * i] = hs[u][3 * i + 1];
                hs[u][3 * i + 1] = hs[u][3 * i + 2];
                hs[u][3 * i + 2] = xt[u][i];
            }
            float4 *sp = reinterpret_cast<float4 *>(state + ((size_t)n * D + c0) * 3);
#pragma unroll
            for (int j = 0; j < 6; ++j)
                sp[j] = make_float4(hs[u][4 * j], hs[u][4 * j + 1], hs[u][4 * j + 2], hs[u][4 * j + 3]);
            Vec8<T>::store(y + (size_t)n * D + c0, out);
        }
    }
}

}  // namespace

bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base, uint64_t cols,
                 uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);

// CTAs of the prefill kernel an SM holds at once (looked up once per device and element type)
template <typename T>
static int resident_ctas(size_t bytes) {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) dev = -1;
    if (dev >= 0) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv_prefill_kernel<T>, kCvThreads, bytes) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        return 1;
    }
    if (dev >= 0) cache[dev].store(per_sm, std::memory_order_relaxed);
    return per_sm;
}

template <typename T>
static int conv_prefill(const T *x, const float *w, const float *b, const float *st_in, float *st_out, T *y, int nseq,
                        int Tlen, int D, const int32_t *cu, cudaStream_t st) {
    const int64_t rows = cu ? (int64_t)Tlen : (int64_t)nseq * Tlen;
    if (rows >= (1ll << 31) - kCvTile) return GLA_ERR_UNSUPPORTED;
    if (rows > 0) {
        const int slab = D < kCvSlab ? D : kCvSlab;  // a multiple of 8 (D % 8 == 0)
        const int64_t nslabs = (D + slab - 1) / slab;
        const int64_t ntiles = (rows + kCvTile - 1) / kCvTile;
        if (nslabs > 65535) return GLA_ERR_UNSUPPORTED;
        CUtensorMap m;
        const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        if (!make_map_2d(&m, dt, (uint32_t)sizeof(T), x, (uint64_t)D, (uint64_t)rows, (uint32_t)slab, kCvBoxRows,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return GLA_ERR_LAUNCH;
        constexpr int NST = CvStages<T>::n;
        const size_t bytes = (size_t)NST * kCvBoxRows * slab * sizeof(T) + 16 * NST + 16;
        if (cudaFuncSetAttribute(conv_prefill_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
            cudaSuccess)
            return GLA_ERR_LAUNCH;
        // one wave: as many CTAs as the SMs hold at once (rounded down to whole slabs), each walking tiles
        // t, t + gridDim.x, ...; a second partial wave would double the time of its tiles.  At any moment the
        // CTAs of all slabs read about the same rows, so DRAM sees whole rows of x (contiguous tile ranges
        // per CTA over all SMs measured slower)
        const int per_sm = resident_ctas<T>(bytes);
        int64_t gx = (int64_t)per_sm * device_info().sm_count / nslabs;
        gx = gx < 1 ? 1 : gx;
        gx = gx < ntiles ? gx : ntiles;
        dim3 grid((unsigned)gx, (unsigned)nslabs);
        conv_prefill_kernel<T><<<grid, kCvThreads, bytes, st>>>(m, w, b, st_in, st_out, y, rows, nseq, Tlen, D, slab,
                                                                cu, ntiles);
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

// blocks of the step kernel the device holds at once (looked up once per device; 0 if that failed)
static int step_resident_blocks() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv_step_kernel<__nv_bfloat16>, kStepThreads, 0) !=
            cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        return 0;
    }
    cache[dev].store(per_sm * device_info().sm_count, std::memory_order_relaxed);
    return per_sm * device_info().sm_count;
}

int conv1d_silu_step_bf16(const void *x, const float *w, const float *b, float *state, void *y, int N, int D,
                          cudaStream_t st) {
    using B = __nv_bfloat16;
    const int cgroups = (D / kVec + kStepThreads - 1) / kStepThreads;
    if (N <= 0) return GLA_OK;
    // sequences per block: the fewest that keep the grid within one wave
    const int resident = step_resident_blocks();
    int spb = kStepSeqs;
    if (resident > 0) {
        const int64_t per_wave = resident / cgroups;  // blocks of sequences per wave
        spb = per_wave > 0 ? (int)(((int64_t)N + per_wave - 1) / per_wave) : N;
    }
    const int ngroups = (N + spb - 1) / spb;
    if (ngroups > 65535) return GLA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)cgroups, (unsigned)ngroups);
    conv_step_kernel<B><<<grid, kStepThreads, 0, st>>>((const B *)x, w, b, state, (B *)y, N, D, spb);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

}  // namespace gla
