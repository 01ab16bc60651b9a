// gla_simt.cu — chunkwise Simple GLA forward on the CUDA cores (f32 FMA).
//
// Serves f32 inputs (where the tensor-core path's bf16 operands would not meet
// an f32 accuracy bar) and bf16 shapes outside the tensor-core kernel's
// envelope.  One CTA owns one (sequence, head) chain and one tile of dv
// columns, and walks the chain's chunks in order with the state tile resident
// in shared memory (columns of the state are independent: column block J of S
// only ever meets column block J of v).
//
// Per chunk c of length L (page "线性注意力模型如何实现固定推理状态", section
// "挑战 1": masked intra-chunk linear attention plus the carried state, then the
// chunk state update; Figure 3):
//   A   = (Q K^T) .* D,          D_ij = lambda^(i-j) for j <= i else 0
//   O   = A V + diag(lambda^(i+1)) Q S
//   S   = lambda^L S + K^T diag(lambda^(L-1-j)) V
//
// The same kernel runs the three recurrences of the backward pass (the page's
// section "挑战 3": the backward differentiates every sequential state update).
// With G_t = dL/dS_t, G_t = lambda G_{t+1} + q_t^T do_t and G_T = dhT, the
// gradients are dq_t = do_t S_t^T, dk_t = v_t G_t^T, dv_t = k_t G_t and
// dh0 = lambda G_1.  Each is a GLA-type recurrence with roles exchanged:
//   dv: reversed time, q' = k, k' = q, v' = do, initial state dhT
//   dk: reversed time, q' = v, k' = do, v' = q, initial state dhT^T
//   dq: forward time,  q' = do, k' = v, v' = k, initial state h0^T
// so the kernel takes a time direction, an initial state read transposed, an
// initial state that enters without the first step's decay (G_T = dhT is not
// decayed before q_T^T do_T is added) and a final state scaled by lambda.
#include <algorithm>

#include "gla_common.cuh"

GLA_DEFINE_STATUS(simt)

namespace gla {
namespace {

constexpr int kThreads = 256;

struct SimtSmem {
    int dkp, dvtp, cp;
    size_t q, k, vv, a, s, tab, total;  // float offsets
};

__host__ __device__ inline SimtSmem simt_layout(int C, int dk, int dvt) {
    SimtSmem L;
    L.dkp = dk + 1;
    L.dvtp = dvt + 4;
    L.cp = C + 1;
    L.q = 0;
    L.k = L.q + (size_t)C * L.dkp;
    L.vv = L.k + (size_t)C * L.dkp;
    L.a = L.vv + (size_t)C * L.dvtp;
    L.s = L.a + (size_t)C * L.cp;
    L.tab = L.s + (size_t)dk * dvt;
    L.total = L.tab + C + 4;
    return L;
}

// Initial / final state handling for the backward's recurrences (all zero for the forward).
enum : int {
    kH0Transposed = 1,  // h0 is stored [dv][dk] per chain: S[d][c] = h0[c][d]
    kH0Undecayed = 2,   // h0 enters the first step without its decay: S_1 = h0 + k_1^T v_1
    kHTTimesDecay = 4,  // hT is written as lambda * S_T
    kStrongOnly = 8,    // only heads with log_decay < -0.3 (the others are left untouched)
};

template <typename T, int C, bool Rev>
__global__ void __launch_bounds__(kThreads)
simt_chunk_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                  const float *__restrict__ log_decay, const float *__restrict__ h0,
                  T *__restrict__ out, float *__restrict__ hT, int nseq, int Tlen, int H, int dk,
                  int dv, int dvt, const int32_t *__restrict__ cu, int state_mode, const T *__restrict__ gate,
                  int gate_kind) {
    extern __shared__ float smem[];
    const SimtSmem Lo = simt_layout(C, dk, dvt);
    float *Qs = smem + Lo.q, *Ks = smem + Lo.k, *Vs = smem + Lo.vv, *As = smem + Lo.a;
    float *Ss = smem + Lo.s, *tab = smem + Lo.tab;
    const int dkp = Lo.dkp, dvtp = Lo.dvtp, cp = Lo.cp;

    const int chain = blockIdx.x;
    const int s = chain / H, h = chain % H;
    const int j0 = blockIdx.y * dvt;
    const int nc = min(dvt, dv - j0);  // valid columns in this tile
    const int tid = threadIdx.x;

    SeqRange r;
    if (!seq_range(s, Tlen, cu, r)) {
        if (tid == 0) record_status(GLA_ERR_DEVICE_ARG);
        return;
    }

    // powers of lambda: tab[n] = lambda^n, n = 0..C
    const float ld = __ldg(log_decay + h);
    if ((state_mode & kStrongOnly) && ld >= -0.3f) return;  // served by the tensor-core backward
    for (int n = tid; n <= C; n += kThreads) tab[n] = expf((float)n * ld);

    // state tile: S[d][c] for c < dvt (columns beyond nc kept at zero)
    const size_t sbase = ((size_t)s * H + h) * dk * dv;
    const bool h0t = (state_mode & kH0Transposed) != 0;
    for (int e = tid; e < dk * dvt; e += kThreads) {
        const int d = e / dvt, c = e % dvt;
        const size_t off = h0t ? (size_t)(j0 + c) * dk + d : (size_t)d * dv + j0 + c;
        Ss[e] = (h0 != nullptr && c < nc) ? __ldg(h0 + sbase + off) : 0.f;
    }
    // token row of chunk-local position i in the chunk that starts c0 tokens into the walk
    auto row_of = [&](int64_t c0, int i) -> int64_t {
        return Rev ? r.start + r.len - 1 - (c0 + i) : r.start + c0 + i;
    };

    for (int64_t c0 = 0; c0 < r.len; c0 += C) {
        const int L = (r.len - c0 < (int64_t)C) ? (int)(r.len - c0) : C;
        // decay exponents of the carried-state terms are one lower in the first chunk when the
        // initial state enters undecayed
        const int sh = (c0 == 0 && (state_mode & kH0Undecayed)) ? 1 : 0;
        __syncthreads();
        // ---- load the chunk (rows >= L are zero) ----
        for (int e = tid; e < C * dk; e += kThreads) {
            const int i = e / dk, d = e % dk;
            float qv = 0.f, kv = 0.f;
            if (i < L) {
                const size_t off = ((size_t)row_of(c0, i) * H + h) * dk + d;
                qv = to_f32(q[off]);
                kv = to_f32(k[off]);
            }
            Qs[i * dkp + d] = qv;
            Ks[i * dkp + d] = kv;
        }
        for (int e = tid; e < C * dvt; e += kThreads) {
            const int i = e / dvt, c = e % dvt;
            float vv = 0.f;
            if (i < L && c < nc) vv = to_f32(v[((size_t)row_of(c0, i) * H + h) * dv + j0 + c]);
            Vs[i * dvtp + c] = vv;
        }
        __syncthreads();
        // ---- A = (Q K^T) .* D, 4x4 register tiles ----
        for (int blk = tid; blk < (C / 4) * (C / 4); blk += kThreads) {
            const int bi = blk / (C / 4), bj = blk % (C / 4);
            float acc[4][4] = {};
            if (bj <= bi) {
                for (int d = 0; d < dk; ++d) {
                    float qa[4], kb[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) qa[a] = Qs[(bi * 4 + a) * dkp + d];
#pragma unroll
                    for (int b = 0; b < 4; ++b) kb[b] = Ks[(bj * 4 + b) * dkp + d];
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qa[a], kb[b], acc[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int i = bi * 4 + a, j = bj * 4 + b;
                    As[i * cp + j] = (j <= i) ? acc[a][b] * tab[i - j] : 0.f;
                }
        }
        __syncthreads();
        // ---- O = A V + diag(lambda^(i+1)) Q S ----
        for (int blk = tid; blk < (C / 4) * (dvt / 4); blk += kThreads) {
            const int bi = blk / (dvt / 4), bc = blk % (dvt / 4);
            float inter[4][4] = {}, intra[4][4] = {};
            for (int d = 0; d < dk; ++d) {
                float qa[4], sb[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) qa[a] = Qs[(bi * 4 + a) * dkp + d];
#pragma unroll
                for (int b = 0; b < 4; ++b) sb[b] = Ss[d * dvt + bc * 4 + b];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) inter[a][b] = fmaf(qa[a], sb[b], inter[a][b]);
            }
            const int jmax = min(bi * 4 + 4, L);
            for (int j = 0; j < jmax; ++j) {
                float aa[4], vb[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) aa[a] = As[(bi * 4 + a) * cp + j];
#pragma unroll
                for (int b = 0; b < 4; ++b) vb[b] = Vs[j * dvtp + bc * 4 + b];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) intra[a][b] = fmaf(aa[a], vb[b], intra[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = bi * 4 + a;
                if (i >= L) continue;
                const float g = tab[i + 1 - sh];
                const size_t ro = ((size_t)row_of(c0, i) * H + h) * dv + j0;
                T *orow = out + ro;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int c = bc * 4 + b;
                    if (c < nc) {
                        float o = fmaf(g, inter[a][b], intra[a][b]);
                        if (gate != nullptr) o *= gate_factor(to_f32(gate[ro + c]), gate_kind);
                        orow[c] = from_f32<T>(o);
                    }
                }
            }
        }
        __syncthreads();
        // ---- S = lambda^L S + K^T diag(lambda^(L-1-j)) V ----
        const float gL = tab[L - sh];
        for (int blk = tid; blk < (dk / 4) * (dvt / 4); blk += kThreads) {
            const int bd = blk / (dvt / 4), bc = blk % (dvt / 4);
            float acc[4][4] = {};
            for (int j = 0; j < L; ++j) {
                const float w = tab[L - 1 - j];
                float ka[4], vb[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) ka[a] = Ks[j * dkp + bd * 4 + a] * w;
#pragma unroll
                for (int b = 0; b < 4; ++b) vb[b] = Vs[j * dvtp + bc * 4 + b];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(ka[a], vb[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float &sv = Ss[(bd * 4 + a) * dvt + bc * 4 + b];
                    sv = fmaf(gL, sv, acc[a][b]);
                }
        }
    }
    __syncthreads();
    if (hT != nullptr) {
        // dh0 = lambda G_1; an empty sequence has no step, so its dh0 is dhT itself
        const float gT = ((state_mode & kHTTimesDecay) && r.len > 0) ? tab[1] : 1.f;
        for (int e = tid; e < dk * dvt; e += kThreads) {
            const int d = e / dvt, c = e % dvt;
            if (c < nc) hT[sbase + (size_t)d * dv + j0 + c] = gT * Ss[e];
        }
    }
}

template <typename T, int C, bool Rev>
int launch_c(const T *q, const T *k, const T *v, const float *ld, const float *h0, T *out, float *hT,
             int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu, int state_mode, cudaStream_t st,
             const T *gate, int gate_kind) {
    const DeviceInfo &di = device_info();
    const size_t limit = std::min<size_t>((size_t)di.max_smem_optin, 200 * 1024);
    int dvt = 64;
    while (dvt > dv && dvt > 8) dvt /= 2;
    if (dvt < dv && dv % 8 == 0 && dv < 64) dvt = dv;
    size_t bytes = simt_layout(C, dk, dvt).total * sizeof(float);
    while (bytes > limit && dvt > 8) {
        dvt = std::max(8, (dvt / 2) & ~7);
        bytes = simt_layout(C, dk, dvt).total * sizeof(float);
    }
    if (bytes > limit) return GLA_ERR_UNSUPPORTED;
    auto kern = simt_chunk_kernel<T, C, Rev>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return GLA_ERR_LAUNCH;
    const long long chains = (long long)nseq * H;
    const int tiles = (dv + dvt - 1) / dvt;
    if (chains > 0x7fffffffLL || tiles > 65535) return GLA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)chains, (unsigned)tiles);
    kern<<<grid, kThreads, bytes, st>>>(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, dvt, cu, state_mode, gate,
                                        gate_kind);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

template <typename T, bool Rev = false>
int launch_simt(const T *q, const T *k, const T *v, const float *ld, const float *h0, T *out, float *hT,
                int nseq, int Tlen, int H, int dk, int dv, int chunk, const int32_t *cu, cudaStream_t st,
                int state_mode = 0, const T *gate = nullptr, int gate_kind = 0) {
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return GLA_ERR_UNSUPPORTED;
    // A chunk whose tiles do not fit in shared memory is processed as sub-chunks
    // of half the length (the chunked form is the same map for any chunk length).
    int rc = GLA_ERR_UNSUPPORTED;
    for (int c = chunk; c >= 16 && rc == GLA_ERR_UNSUPPORTED; c /= 2) {
        switch (c) {
            case 16: rc = launch_c<T, 16, Rev>(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, cu, state_mode, st, gate, gate_kind); break;
            case 32: rc = launch_c<T, 32, Rev>(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, cu, state_mode, st, gate, gate_kind); break;
            case 64: rc = launch_c<T, 64, Rev>(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, cu, state_mode, st, gate, gate_kind); break;
            default: rc = launch_c<T, 128, Rev>(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, cu, state_mode, st, gate, gate_kind); break;
        }
    }
    return rc;
}

}  // namespace

int simt_chunk_fwd_f32(const float *q, const float *k, const float *v, const float *ld, const float *h0,
                       float *out, float *hT, int nseq, int Tlen, int H, int dk, int dv, int chunk,
                       const int32_t *cu, cudaStream_t st) {
    return launch_simt<float>(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, chunk, cu, st);
}

int simt_chunk_fwd_bf16(const void *q, const void *k, const void *v, const float *ld, const float *h0,
                        void *out, float *hT, int nseq, int Tlen, int H, int dk, int dv, int chunk,
                        const int32_t *cu, cudaStream_t st) {
    using B = __nv_bfloat16;
    return launch_simt<B>((const B *)q, (const B *)k, (const B *)v, ld, h0, (B *)out, hT, nseq, Tlen, H, dk,
                          dv, chunk, cu, st);
}

// The same forward with the output gate applied to every output row (gate: [rows, H, dv] like out).
int simt_chunk_fwd_gated_bf16(const void *q, const void *k, const void *v, const void *g, int gate_kind,
                              const float *ld, const float *h0, void *out, float *hT, int nseq, int Tlen, int H,
                              int dk, int dv, int chunk, const int32_t *cu, cudaStream_t st) {
    using B = __nv_bfloat16;
    return launch_simt<B>((const B *)q, (const B *)k, (const B *)v, ld, h0, (B *)out, hT, nseq, Tlen, H, dk,
                          dv, chunk, cu, st, 0, (const B *)g, gate_kind);
}

// Backward of the chunked forward: three recurrences (see the top of this file), each a launch of
// the chunk kernel.  dq, dk: [rows, H, dk]; dv: [rows, H, dv]; dh0: [nseq, H, dk, dv] or null;
// dhT: [nseq, H, dk, dv] or null (zero); h0 as in the forward.
template <typename T>
int simt_bwd(const T *q, const T *k, const T *v, const T *dout, const float *ld, const float *h0, const float *dhT,
             T *dq, T *dk_, T *dv_, float *dh0, int nseq, int Tlen, int H, int dk, int dv, int chunk,
             const int32_t *cu, cudaStream_t st, int extra = 0) {
    int rc = launch_simt<T, true>(k, q, dout, ld, dhT, dv_, dh0, nseq, Tlen, H, dk, dv, chunk, cu, st,
                                  kH0Undecayed | kHTTimesDecay | extra);
    if (rc != GLA_OK) return rc;
    rc = launch_simt<T, true>(v, dout, q, ld, dhT, dk_, nullptr, nseq, Tlen, H, dv, dk, chunk, cu, st,
                              kH0Undecayed | kH0Transposed | extra);
    if (rc != GLA_OK) return rc;
    return launch_simt<T, false>(dout, v, k, ld, h0, dq, nullptr, nseq, Tlen, H, dv, dk, chunk, cu, st,
                                 kH0Transposed | extra);
}

int simt_chunk_bwd_f32(const float *q, const float *k, const float *v, const float *dout, const float *ld,
                       const float *h0, const float *dhT, float *dq, float *dk_, float *dv_, float *dh0, int nseq,
                       int Tlen, int H, int dk, int dv, int chunk, const int32_t *cu, cudaStream_t st) {
    return simt_bwd<float>(q, k, v, dout, ld, h0, dhT, dq, dk_, dv_, dh0, nseq, Tlen, H, dk, dv, chunk, cu, st);
}

// The SIMT backward for the heads with log_decay < -0.3 only (companion of the tensor-core backward).
int simt_chunk_bwd_bf16_strong(const void *q, const void *k, const void *v, const void *dout, const float *ld,
                               const float *h0, const float *dhT, void *dq, void *dk_, void *dv_, float *dh0,
                               int nseq, int Tlen, int H, int dk, int dv, int chunk, const int32_t *cu,
                               cudaStream_t st) {
    using B = __nv_bfloat16;
    return simt_bwd<B>((const B *)q, (const B *)k, (const B *)v, (const B *)dout, ld, h0, dhT, (B *)dq, (B *)dk_,
                       (B *)dv_, dh0, nseq, Tlen, H, dk, dv, chunk, cu, st, kStrongOnly);
}

int simt_chunk_bwd_bf16(const void *q, const void *k, const void *v, const void *dout, const float *ld,
                        const float *h0, const float *dhT, void *dq, void *dk_, void *dv_, float *dh0, int nseq,
                        int Tlen, int H, int dk, int dv, int chunk, const int32_t *cu, cudaStream_t st) {
    using B = __nv_bfloat16;
    return simt_bwd<B>((const B *)q, (const B *)k, (const B *)v, (const B *)dout, ld, h0, dhT, (B *)dq, (B *)dk_,
                       (B *)dv_, dh0, nseq, Tlen, H, dk, dv, chunk, cu, st);
}

}  // namespace gla
