// gla_tc.cu — chunked Simple GLA forward on the Blackwell tensor cores
// (tcgen05.mma with TMEM accumulators, operands staged by TMA), bf16 in,
// f32 accumulate and f32 state.
//
// The method (page "线性注意力模型如何实现固定推理状态", section "挑战 1", chunked
// GLA and Figure 3): within chunk c of length L, local positions i, j,
//   O_c = ((Q_c K_c^T) .* D) V_c + diag(lambda^(i+1)) Q_c S_{c-1},  D_ij = lambda^(i-j) [j <= i]
//   S_c = lambda^L S_{c-1} + K_c^T diag(lambda^(L-1-j)) V_c
// Only the state chain is sequential; everything inside a chunk is dense
// contraction work.
//
// One CTA owns one (sequence, head) chain and walks its 128-token chunks in
// order with the f32 state resident in TMEM for the whole chain.  Per chunk the
// four contractions are tcgen05.mma instructions (M = 128, K-steps of 16):
//   MMA1  A    = Q K^T                      TMEM cols [384, 512)   A: Q (smem), B: K (smem)
//   MMA3  O    = (diag(lambda^(i+1)) Q) S   TMEM cols [0, dv)      A: Q' (smem), B: S bf16 (smem)
//   MMA4  S   += (diag(lambda^(L-1-j)) K)^T V  TMEM cols [192, 192+dv)  A: K'^T (smem), B: V (smem)
//   MMA2  O   += P V,  P = bf16(A .* D)     A: P (TMEM, aliases A), B: V (smem)
// The state rows are dk (<= 128), padded to M = 128; rows >= dk of the state
// accumulator are never read.
//
// Warp roles (320 threads):
//   warps 0-7  "compute": two warpgroups; thread t owns TMEM lane t % 128 (a
//              token row of A/P/O, a dk row of S) and half of the columns.
//              Per chunk: state pass (read S_{c-1} from TMEM, write its bf16
//              copy for MMA3, pre-scale it by lambda^L for MMA4), decay of Q
//              and K rows in place, decay mask A -> P, output epilogue.
//   warp 8     TMA producer: Q (single buffer), K and V (double buffer).
//   warp 9     MMA issuer and TMEM owner.
// Hand-offs are mbarriers; every wait is bounded (see sm100_ptx.cuh) and a
// timeout is recorded as GLA_ERR_TIMEOUT in the device status word.
//
// Shared-memory operand layouts (all TMA-compatible, bf16):
//   Q, K tiles   [128 tokens][dk], 64-byte swizzle, one atom per 32 dk columns
//                (atom = 128 rows x 64 B = 8 KB).  K-major operand for MMA1/MMA3;
//                read as the MN-major A operand K'^T of MMA4.
//   V tiles      [128 tokens][dv], 128-byte swizzle, atoms of 64 dv columns
//                (128 rows x 128 B = 16 KB).  MN-major B operand of MMA2/MMA4.
//   S copy       [dk][dv] bf16, 128-byte swizzle, atoms of 64 dv columns
//                (dk rows x 128 B).  MN-major B operand of MMA3.
#include <mutex>

#include "gla_common.cuh"
#include "sm100_ptx.cuh"

GLA_DEFINE_STATUS(tc)

namespace gla {
namespace {

using namespace ptx;

constexpr int kC = 128;              // chunk length (MMA M and the token K extent)
constexpr int kThreads = 320;        // 8 compute warps + producer + MMA warp
constexpr int kComputeThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;        // O accumulator  [0, dv)
constexpr uint32_t kColS = 192;      // state          [192, 192 + dv)
constexpr uint32_t kColA = 384;      // A = Q K^T      [384, 512); P aliases [384, 448)
constexpr uint64_t kWaitBudgetNs = 4000000000ull;  // 4 s per wait

struct Params {
    const float *log_decay;
    const float *h0;
    __nv_bfloat16 *out;
    float *hT;
    const int32_t *cu;
    int T, H, dk, dv;
};

// Shared memory plan (bytes from the 1024-aligned base).
struct Smem {
    uint32_t q, k0, k1, v0, v1, s, tab, bars, slot, abort, total;
};

__host__ __device__ inline Smem smem_plan(int dk, int dv) {
    Smem p;
    const uint32_t qk = (uint32_t)(dk / 32) * 8192u;
    const uint32_t vv = (uint32_t)(dv / 64) * 16384u;
    p.q = 0;
    p.k0 = p.q + qk;
    p.k1 = p.k0 + qk;
    p.v0 = p.k1 + qk;  // MMA4 reads up to 4 atoms from a K tile: V follows, so the over-read stays in bounds
    p.v1 = p.v0 + vv;
    p.s = p.v1 + vv;
    p.tab = p.s + (uint32_t)dk * 128u * (uint32_t)(dv / 64);
    p.bars = p.tab + 132 * 4;
    p.bars = (p.bars + 7u) & ~7u;
    p.slot = p.bars + 16 * 8;
    p.abort = p.slot + 4;
    p.total = p.abort + 4;
    return p;
}

// barrier indices
enum { B_QFULL = 0, B_QEMPTY, B_KVFULL0, B_KVFULL1, B_KVEMPTY0, B_KVEMPTY1, B_AFULL, B_PREP, B_SREADY, B_PFULL,
       B_OFULL, B_OFREE, B_SFULL, B_FINAL, B_COUNT };

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void scale_row_bf16(uint8_t *row, int nbytes, float f) {
    // nbytes is a multiple of 16; rows keep their 16-byte chunks whatever the swizzle
    for (int b = 0; b < nbytes; b += 16) {
        uint4 x = *reinterpret_cast<uint4 *>(row + b);
        uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&w[e]);
            float2 fl = __bfloat1622float2(h);
            w[e] = pack_bf16x2(fl.x * f, fl.y * f);
        }
        *reinterpret_cast<uint4 *>(row + b) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
gla_tc_chunk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int dk = P.dk, dv = P.dv, H = P.H;
    const Smem sp = smem_plan(dk, dv);
    const uint32_t sbase = smem_u32(smem);
    float *tab = reinterpret_cast<float *>(smem + sp.tab);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + sp.slot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + sp.abort);
    auto bar = [&](int i) -> uint32_t { return sbase + sp.bars + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chain = blockIdx.x;
    const int seq = chain / H, h = chain % H;

    SeqRange rng;
    const bool valid = seq_range(seq, P.T, P.cu, rng);
    const int64_t len = valid ? rng.len : 0;
    const int nchunks = (int)((len + kC - 1) / kC);
    const int row0 = (int)rng.start;
    const float ld = __ldg(P.log_decay + h);

    if (threadIdx.x == 0) {
        if (!valid) record_status(GLA_ERR_DEVICE_ARG);
        *abort_flag = 0;
        mbar_init(bar(B_QFULL), 1);
        mbar_init(bar(B_QEMPTY), 1);
        mbar_init(bar(B_KVFULL0), 1);
        mbar_init(bar(B_KVFULL1), 1);
        mbar_init(bar(B_KVEMPTY0), 1);
        mbar_init(bar(B_KVEMPTY1), 1);
        mbar_init(bar(B_AFULL), 1);
        mbar_init(bar(B_PREP), kComputeThreads);
        mbar_init(bar(B_SREADY), kComputeThreads);
        mbar_init(bar(B_PFULL), kComputeThreads);
        mbar_init(bar(B_OFULL), 1);
        mbar_init(bar(B_OFREE), kComputeThreads);
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_FINAL), 1);
        fence_mbar_init();
    }
    if (threadIdx.x < kC + 4) tab[threadIdx.x] = (threadIdx.x <= kC) ? expf((float)threadIdx.x * ld) : 0.f;
    if (warp == kMmaWarp) {
        tmem_alloc(sbase + sp.slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (!valid) {
        // nothing to compute; hT for an invalid sequence is left untouched
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && nchunks > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const int nka = dk / 32, nva = dv / 64;
            const uint32_t kvbytes = (uint32_t)nka * 8192u + (uint32_t)nva * 16384u;
            const uint32_t qbytes = (uint32_t)nka * 8192u;
            bool ok = true;
            for (int c = 0; c < nchunks && ok; ++c) {
                const int s = c & 1;
                const int y = row0 + c * kC;
                if (c >= 2) ok = mbar_wait(bar(B_KVEMPTY0 + s), ((c >> 1) - 1) & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                mbar_expect_tx(bar(B_KVFULL0 + s), kvbytes);
                const uint32_t kdst = sbase + (s ? sp.k1 : sp.k0), vdst = sbase + (s ? sp.v1 : sp.v0);
                for (int a = 0; a < nka; ++a) tma_load_2d(kdst + a * 8192u, &tmK, h * dk + 32 * a, y, bar(B_KVFULL0 + s));
                for (int a = 0; a < nva; ++a) tma_load_2d(vdst + a * 16384u, &tmV, h * dv + 64 * a, y, bar(B_KVFULL0 + s));
                if (c >= 1) ok = mbar_wait(bar(B_QEMPTY), (c - 1) & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                mbar_expect_tx(bar(B_QFULL), qbytes);
                for (int a = 0; a < nka; ++a) tma_load_2d(sbase + sp.q + a * 8192u, &tmQ, h * dk + 32 * a, y, bar(B_QFULL));
            }
            if (!ok) {
                record_status(GLA_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nchunks > 0) {
            const uint32_t id_qk = idesc_bf16(kC, kC, 0, 0);
            const uint32_t id_qs = idesc_bf16(kC, dv, 0, 1);
            const uint32_t id_pv = idesc_bf16(kC, dv, 0, 1);
            const uint32_t id_kv = idesc_bf16(kC, dv, 1, 1);
            const int ksteps_dk = dk / 16;
            bool ok = true;
            for (int c = 0; c < nchunks && ok; ++c) {
                const int s = c & 1;
                const uint32_t kbuf = sbase + (s ? sp.k1 : sp.k0), vbuf = sbase + (s ? sp.v1 : sp.v0);
                const uint32_t qbuf = sbase + sp.q, sbuf = sbase + sp.s;
                ok = mbar_wait(bar(B_KVFULL0 + s), (c >> 1) & 1, abort_flag, kWaitBudgetNs) &&
                     mbar_wait(bar(B_QFULL), c & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
                // MMA1: A = Q K^T (both K-major, 64B swizzle; 2 K-steps per 32-column atom)
                for (int kk = 0; kk < ksteps_dk; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 1) * 8192u + (uint32_t)(kk & 1) * 32u;
                    mma_ss(tmem + kColA, smem_desc(qbuf + off, 16, 512, kSwizzle64B),
                           smem_desc(kbuf + off, 16, 512, kSwizzle64B), id_qk, kk > 0);
                }
                mma_commit(bar(B_AFULL));
                ok = mbar_wait(bar(B_PREP), c & 1, abort_flag, kWaitBudgetNs) &&
                     mbar_wait(bar(B_SREADY), c & 1, abort_flag, kWaitBudgetNs) &&
                     (c == 0 || mbar_wait(bar(B_OFREE), (c - 1) & 1, abort_flag, kWaitBudgetNs));
                if (!ok) break;
                tc_fence_after();
                // MMA3: O = Q' S_{c-1} (A K-major 64B swizzle; B = S copy, MN-major 128B swizzle)
                for (int kk = 0; kk < ksteps_dk; ++kk) {
                    const uint32_t aoff = (uint32_t)(kk >> 1) * 8192u + (uint32_t)(kk & 1) * 32u;
                    mma_ss(tmem + kColO, smem_desc(qbuf + aoff, 16, 512, kSwizzle64B),
                           smem_desc(sbuf + (uint32_t)kk * 2048u, (uint32_t)dk * 128u, 1024, kSwizzle128B), id_qs,
                           kk > 0);
                }
                // MMA4: S += K'^T V (A MN-major 64B swizzle over dk, B MN-major 128B swizzle over dv)
                for (int kk = 0; kk < kC / 16; ++kk) {
                    mma_ss(tmem + kColS, smem_desc(kbuf + (uint32_t)kk * 1024u, 8192, 512, kSwizzle64B),
                           smem_desc(vbuf + (uint32_t)kk * 2048u, 16384, 1024, kSwizzle128B), id_kv, 1);
                }
                mma_commit(bar(B_SFULL));
                mma_commit(bar(B_QEMPTY));
                ok = mbar_wait(bar(B_PFULL), c & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
                // MMA2: O += P V (A = P in TMEM, 8 columns per K-step of 16 tokens)
                for (int kk = 0; kk < kC / 16; ++kk) {
                    mma_ts(tmem + kColO, tmem + kColA + (uint32_t)kk * 8u,
                           smem_desc(vbuf + (uint32_t)kk * 2048u, 16384, 1024, kSwizzle128B), id_pv, 1);
                }
                mma_commit(bar(B_OFULL));
                mma_commit(bar(B_KVEMPTY0 + s));
            }
            if (!ok) {
                record_status(GLA_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ compute warps
        const int t = threadIdx.x;          // 0..255
        const int wg = t >> 7;              // column half
        const int r = t & 127;              // TMEM lane = token row / state row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int half_dv = dv / 2;
        const int64_t hstate = ((int64_t)seq * H + h) * dk * dv;
        bool ok = true;
        for (int c = 0; c <= nchunks && ok; ++c) {
            const int Lc = (c < nchunks) ? (int)((len - (int64_t)c * kC < kC) ? (len - (int64_t)c * kC) : kC) : 0;
            // ---- state pass: S_{c-1} -> bf16 copy for MMA3, pre-scaled by lambda^L_c for MMA4 (or hT) ----
            if (c >= 1) {
                ok = mbar_wait(bar(B_SFULL), (c - 1) & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
            }
            const bool last = (c == nchunks);
            const float g = last ? 1.f : tab[Lc];
            if (r < dk) {
                for (int j0 = wg * half_dv; j0 < (wg + 1) * half_dv; j0 += 32) {
                    uint32_t v[32];
                    if (c >= 1) {
                        tmem_ld32(tmem + lane_base + kColS + (uint32_t)j0, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(P.h0 ? __ldg(P.h0 + hstate + (int64_t)r * dv + j0 + e) : 0.f);
                    }
                    if (last) {
                        if (P.hT) {
                            float4 *dst = reinterpret_cast<float4 *>(P.hT + hstate + (int64_t)r * dv + j0);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                     __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                        }
                        continue;
                    }
                    // bf16 copy into the MN-major, 128B-swizzled S tile
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const int j = j0 + 8 * q8;
                        const uint32_t atom = (uint32_t)(j >> 6), chunk16 = (uint32_t)((j & 63) >> 3);
                        uint8_t *dst = smem + sp.s + atom * (uint32_t)dk * 128u + (uint32_t)r * 128u +
                                       ((chunk16 ^ (uint32_t)(r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 0]), __uint_as_float(v[8 * q8 + 1])),
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 2]), __uint_as_float(v[8 * q8 + 3])),
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 4]), __uint_as_float(v[8 * q8 + 5])),
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 6]), __uint_as_float(v[8 * q8 + 7])));
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * g);
                    tmem_st32(tmem + lane_base + kColS + (uint32_t)j0, v);
                }
            }
            if (last) break;
            tmem_wait_st();
            fence_async_shared();
            tc_fence_before();
            mbar_arrive(bar(B_SREADY));

            // ---- decay Q and K rows in place (after MMA1 has read them) ----
            ok = mbar_wait(bar(B_AFULL), c & 1, abort_flag, kWaitBudgetNs);
            if (!ok) break;
            tc_fence_after();
            {
                const int s = c & 1;
                const int nka = dk / 32;
                if (wg == 0) {
                    const float f = tab[min(r + 1, kC)];
                    for (int a = 0; a < nka; ++a) scale_row_bf16(smem + sp.q + a * 8192 + r * 64, 64, f);
                } else {
                    const float f = (r < Lc) ? tab[Lc - 1 - r] : 0.f;
                    uint8_t *kb = smem + (s ? sp.k1 : sp.k0);
                    for (int a = 0; a < nka; ++a) scale_row_bf16(kb + a * 8192 + r * 64, 64, f);
                }
            }
            fence_async_shared();
            mbar_arrive(bar(B_PREP));

            // ---- decay mask: P = bf16(A .* D), written over the first half of A's columns ----
            {
                uint32_t a0[32], a1[32];
                const uint32_t acol = kColA + (uint32_t)(64 * wg);
                tmem_ld32(tmem + lane_base + acol, a0);
                tmem_ld32(tmem + lane_base + acol + 32, a1);
                tmem_wait_ld();
                uint32_t p[32];
                const bool row_ok = r < Lc;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = 64 * wg + 2 * e;
                    const int d0 = r - j, d1 = r - j - 1;
                    const float f0 = (row_ok && d0 >= 0) ? tab[max(d0, 0)] : 0.f;
                    const float f1 = (row_ok && d1 >= 0) ? tab[max(d1, 0)] : 0.f;
                    p[e] = pack_bf16x2(__uint_as_float(a0[2 * e]) * f0, __uint_as_float(a0[2 * e + 1]) * f1);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = 64 * wg + 32 + 2 * e;
                    const int d0 = r - j, d1 = r - j - 1;
                    const float f0 = (row_ok && d0 >= 0) ? tab[max(d0, 0)] : 0.f;
                    const float f1 = (row_ok && d1 >= 0) ? tab[max(d1, 0)] : 0.f;
                    p[16 + e] = pack_bf16x2(__uint_as_float(a1[2 * e]) * f0, __uint_as_float(a1[2 * e + 1]) * f1);
                }
                // every compute thread has read its A columns before any P column is written
                named_bar_sync(1, kComputeThreads);
                tmem_st32(tmem + lane_base + kColA + (uint32_t)(32 * wg), p);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar(B_PFULL));

            // ---- output epilogue: O (f32, TMEM) -> bf16 rows of out ----
            ok = mbar_wait(bar(B_OFULL), c & 1, abort_flag, kWaitBudgetNs);
            if (!ok) break;
            tc_fence_after();
            {
                __nv_bfloat16 *orow = P.out + ((int64_t)(row0 + (int64_t)c * kC + r) * H + h) * dv;
                for (int j0 = wg * half_dv; j0 < (wg + 1) * half_dv; j0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kColO + (uint32_t)j0, v);
                    tmem_wait_ld();
                    if (r < Lc) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + j0);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(
                                pack_bf16x2(__uint_as_float(v[8 * e + 0]), __uint_as_float(v[8 * e + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_OFREE));
        }
        if (!ok) {
            record_status(GLA_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    // ---- teardown: all roles done; make sure no tensor-core work is in flight, free TMEM ----
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        if (*abort_flag) {
            if (lane == 0) mma_commit(bar(B_FINAL));
            __syncwarp();
            mbar_wait(bar(B_FINAL), 0, nullptr, kWaitBudgetNs);
        }
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side ------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, (cuuint32_t)kC};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_chunk_supported(int dk, int dv, int chunk) {
    if (!(chunk == kC && dk % 32 == 0 && dk >= 32 && dk <= 128 && dv % 64 == 0 && dv >= 64 && dv <= 192))
        return false;
    return smem_plan(dk, dv).total + 1024 <= (uint32_t)device_info().max_smem_optin;
}

int tc_chunk_fwd_bf16(const void *q, const void *k, const void *v, const float *ld, const float *h0, void *out,
                      float *hT, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu, cudaStream_t st) {
    if (!tc_chunk_supported(dk, dv, kC)) return GLA_ERR_UNSUPPORTED;
    const uint64_t rows = cu ? (uint64_t)Tlen : (uint64_t)nseq * (uint64_t)Tlen;
    if (rows >= (1ull << 31)) return GLA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mk, k, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mv, v, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return GLA_ERR_LAUNCH;
    const Smem sp = smem_plan(dk, dv);
    const size_t bytes = sp.total + 1024;  // + alignment slack
    const DeviceInfo &di = device_info();
    if (bytes > (size_t)di.max_smem_optin) return GLA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(gla_tc_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return GLA_ERR_LAUNCH;
    Params p;
    p.log_decay = ld;
    p.h0 = h0;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.hT = hT;
    p.cu = cu;
    p.T = Tlen;
    p.H = H;
    p.dk = dk;
    p.dv = dv;
    const long long chains = (long long)nseq * H;
    if (chains > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    gla_tc_chunk_kernel<<<(unsigned)chains, kThreads, bytes, st>>>(mq, mk, mv, p);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

}  // namespace gla
