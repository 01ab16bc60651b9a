// gla_bwd_tc.cu — gradients of the chunked forward on the Blackwell tensor cores.
//
// The backward of the recurrence (page "线性注意力模型如何实现固定推理状态",
// section "挑战 3": the backward pass differentiates every sequential state
// update) splits into two thin sequential parts and one chunk-parallel part.
// With G_c = dL/dS_c the gradient reaching the state at the end of chunk c
// (G_last = dhT) and S_{c-1} the state before chunk c:
//   state passes (gla_tc.cu, mode kStates): S_{c-1} forwards from h0 and
//     G_{c-1} = lambda^L G_c + sum_i lambda^(i+1) q_i^T do_i backwards from
//     dhT, each stored as a bf16 tile per chunk; dh0 = G before chunk 0.
//   this kernel, one CTA per (chunk, head), no recurrence: within chunk c of
//   length L (local positions i, j), A = Q K^T, B = dO V^T,
//     dQ = diag(lambda^(i+1)) dO S_{c-1}^T + (B .* D) K
//     dK = (B .* D)^T Q + diag(lambda^(L-1-j)) V G_c^T
//     dV = (A .* D)^T dO + diag(lambda^(L-1-j)) K G_c
//   with D_ij = lambda^(i-j) for j <= i.  The decay is factored so that every
//   inter-chunk term shares its accumulator with the intra-chunk term:
//     dV_j = lambda^(L-1-j) [ sum_i A_ij lambda^(i+1-L) do_i + k_j G_c ]
//     dK_j = lambda^(L-1-j) [ sum_i B_ij lambda^(i+1-L) q_i + v_j G_c^T ]
//     dQ_i = lambda^(i+1)   [ sum_j B_ij lambda^-(j+1) k_j + do_i S_{c-1}^T ]
//   so the masks carry a column factor and the epilogues a row factor.  The
//   factors stay far from overflow for lambda >= e^-0.3; CTAs of heads with
//   stronger decays return at once (their gradients come from the chunked SIMT
//   backward, which the host runs for those heads only).
//
// Per CTA (256 threads; warps w and w + 4 share TMEM lane quadrant w, and so row 32 w + lane; the
// masks split each row's 128 score columns between the two, the epilogue its three accumulators):
//   TMA:   Q, K tiles [128 x dk] (64B swizzle), V, dO tiles [128 x dv] (128B
//          swizzle), the two bf16 state tiles as raw images (bulk copies)
//   MMA1   A^T = K Q^T            -> scratch [384, 512)   mask -> P1 (bf16)
//   MMA2   dV  = P1 dO + K G_c    -> [0, dv)
//   MMA3   B^T = V dO^T           -> scratch              mask -> P2
//   MMA4   dK  = P2 Q + V G_c^T   -> [dv, dv+dk)
//   MMA5   B   = dO V^T           -> scratch              mask -> P3
//   MMA6   dQ  = P3 K + dO S^T    -> [dv+dk, dv+2dk)
//   epilogue: row factors, bf16, stores of the rows below L; in a full chunk dV and dK
//          are staged over V and Q and stored while mask 3 and MMA6 run, dQ after MMA6.
#include <mutex>

#include "gla_common.cuh"
#include "sm100_ptx.cuh"

GLA_DEFINE_STATUS(bwd)

namespace gla {

bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              CUtensorMapSwizzle sw, uint32_t box_rows);
int tc_state_pass_bf16(const void *ka, const void *va, const float *ld, const float *init, float *final_,
                       void *images, int reverse, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu,
                       cudaStream_t st);
bool tc_chunk_supported(int dk, int dv, int chunk);
int simt_chunk_bwd_bf16_strong(const void *, const void *, const void *, const void *, const float *, const float *,
                               const float *, void *, void *, void *, float *, int, int, int, int, int, int,
                               const int32_t *, cudaStream_t);

namespace {

using namespace ptx;

constexpr int kC = 128;
constexpr int kThreads = 256;  // two warps per TMEM lane quadrant
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColScratch = 384;
constexpr uint64_t kWaitBudgetNs = 4000000000ull;
constexpr float kFactoredMinLogDecay = -0.3f;

struct BwdParams {
    const float *log_decay;
    const int32_t *cu;
    const __nv_bfloat16 *s_img;  // [slots, H, dk, dv] bf16 tiles: state before each chunk
    const __nv_bfloat16 *g_img;  // [slots, H, dk, dv] bf16 tiles: gradient state at each chunk's end
    __nv_bfloat16 *dq, *dk, *dv;
    int nseq, T, H, dkk, dvv, slots;
};

struct BwdSmem {
    uint32_t q, k, v, dout, s, g, tab, utab, wcol, bars, slot, abort, total;
};

__host__ __device__ inline BwdSmem bwd_plan(int dk, int dv) {
    BwdSmem p;
    const uint32_t qk = (uint32_t)(dk / 32) * 8192u, vv = (uint32_t)(dv / 64) * 16384u, st = (uint32_t)dk * dv * 2u;
    p.q = 0;
    p.k = p.q + qk;
    p.v = p.k + qk;
    p.dout = p.v + vv;
    p.s = p.dout + vv;
    p.g = p.s + st;
    p.tab = p.g + st;
    p.utab = p.tab + 132 * 4;
    p.wcol = p.utab + 128 * 4;
    p.bars = (p.wcol + 128 * 4 + 7u) & ~7u;
    p.slot = p.bars + 8 * 8;
    p.abort = p.slot + 4;
    p.total = p.abort + 4;
    return p;
}

// loads land in three groups so that MMA1 can start on Q, K alone
enum { B_LOAD = 0, B_LOAD2, B_LOAD3, B_MMA, B_MASK, B_FINAL };

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&p)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]), "r"(p[8]),
        "r"(p[9]), "r"(p[10]), "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]), "r"(p[15])
        : "memory");
}

// Mask the 128 x 128 f32 scores in the scratch columns into bf16 P (in place, 64 columns).  Row r
// of this thread; element (r, x) is kept when (lower ? x <= r : x >= r) and both are below L, and
// is multiplied by colf[x].  The two warps of a lane quadrant take score columns [64 half, 64 half + 64)
// each; P block b (16 columns) overwrites score block b / 2, which the other half may still read, so
// every thread holds its scores in registers before the CTA barrier and writes P after it.  The barrier
// is reached by every thread (also when `live` is false: then the warp only passes it).  The kept
// columns of each 32-column block are one 32-bit mask (bit t for column 32 b + t), so no per-element
// comparison is kept live.
// Four f32 values at a 16-byte aligned shared address, as two pairs (values 0, 1 and 2, 3).
__device__ __forceinline__ void lds_f32x2x2(uint32_t addr, uint64_t &a, uint64_t &b) {
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}
// Two f32 values (bit patterns) times the pair g2 with one instruction: mul.rn.f32x2 rounds each lane as
// mul.rn.f32 does, so the results are those of two scalar multiplies.
__device__ __forceinline__ void mul_f32x2(uint32_t &lo, uint32_t &hi, uint64_t g2) {
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%0, %1};\n\tmul.rn.f32x2 t, t, %2;\n\tmov.b64 {%0, %1}, t;\n\t}"
        : "+r"(lo), "+r"(hi)
        : "l"(g2));
}
__device__ __forceinline__ uint64_t f32x2_splat(float g) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(g));
    return d;
}

__device__ __forceinline__ void mask_scores(uint32_t tbase, int r, int L, bool lower, uint32_t colf, int half,
                                            bool live) {
    uint32_t a[2][32];
    if (live) {
        tmem_ld32(tbase + (uint32_t)(64 * half), a[0]);
        tmem_ld32(tbase + (uint32_t)(64 * half + 32), a[1]);
        tmem_wait_ld();
    }
    named_bar_sync(1, kThreads);
    if (!live) return;
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
        const int b = 2 * half + bb;
        const int d = r - 32 * b, lim = L - 32 * b;
        uint32_t bits = lower ? (d >= 31 ? 0xffffffffu : d < 0 ? 0u : (2u << d) - 1u)
                              : (d <= 0 ? 0xffffffffu : d > 31 ? 0u : ~((1u << d) - 1u));
        bits &= lim >= 32 ? 0xffffffffu : lim <= 0 ? 0u : (1u << lim) - 1u;
        if (r >= L) bits = 0u;
        uint32_t p[16];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            uint64_t c01, c23;  // column factors of columns 32 b + 4 g .. + 3 (16-byte aligned table)
            lds_f32x2x2(colf + (uint32_t)(32 * b + 4 * g) * 4u, c01, c23);
            const int e = 2 * g;
            uint32_t x0 = a[bb][2 * e], x1 = a[bb][2 * e + 1], x2 = a[bb][2 * e + 2], x3 = a[bb][2 * e + 3];
            mul_f32x2(x0, x1, c01);
            mul_f32x2(x2, x3, c23);
            p[e] = pack_bf16x2(((bits >> (2 * e)) & 1u) ? __uint_as_float(x0) : 0.f,
                               ((bits >> (2 * e + 1)) & 1u) ? __uint_as_float(x1) : 0.f);
            p[e + 1] = pack_bf16x2(((bits >> (2 * e + 2)) & 1u) ? __uint_as_float(x2) : 0.f,
                                   ((bits >> (2 * e + 3)) & 1u) ? __uint_as_float(x3) : 0.f);
        }
        tmem_st16(tbase + (uint32_t)(16 * b), p);
    }
    tmem_wait_st();
}

// Columns [c_begin, c_end) (multiples of 32) of row r of an accumulator at tcol, times f, as bf16 into a
// staging tile at shared address `tile`, laid out as the TMA box of the output: 64-column atoms of 128-byte
// rows with the 128B swizzle (atom_cols 64), or 32-column atoms of 64-byte rows with the 64B swizzle
// (atom_cols 32).
__device__ __forceinline__ void stage_row(uint32_t tcol, int c_begin, int c_end, float f, int r, uint32_t tile,
                                          int atom_cols) {
    const uint64_t f2 = f32x2_splat(f);
    for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tcol + (uint32_t)c0, a);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) mul_f32x2(a[e], a[e + 1], f2);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t dst;
            if (atom_cols == 64) {
                const uint32_t phys = ((uint32_t)(((c0 & 63) >> 3) + q)) ^ ((uint32_t)r & 7u);
                dst = tile + (uint32_t)(c0 >> 6) * 16384u + (uint32_t)r * 128u + (phys << 4);
            } else {
                const uint32_t phys = (uint32_t)q ^ (((uint32_t)r >> 1) & 3u);
                dst = tile + (uint32_t)(c0 >> 5) * 8192u + (uint32_t)r * 64u + (phys << 4);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                         "r"(pack_bf16x2(__uint_as_float(a[8 * q]), __uint_as_float(a[8 * q + 1]))),
                         "r"(pack_bf16x2(__uint_as_float(a[8 * q + 2]), __uint_as_float(a[8 * q + 3]))),
                         "r"(pack_bf16x2(__uint_as_float(a[8 * q + 4]), __uint_as_float(a[8 * q + 5]))),
                         "r"(pack_bf16x2(__uint_as_float(a[8 * q + 6]), __uint_as_float(a[8 * q + 7])))
                         : "memory");
        }
    }
}

// Row r of an accumulator of `ncols` columns at tcol, times f, as bf16 into dst (global), if r < L.
__device__ __forceinline__ void store_row(uint32_t tcol, int ncols, float f, bool live, __nv_bfloat16 *dst) {
    for (int c0 = 0; c0 < ncols; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tcol + (uint32_t)c0, a);
        tmem_wait_ld();
        if (live) {
            uint4 *d = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                d[q] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * q]) * f, __uint_as_float(a[8 * q + 1]) * f),
                                  pack_bf16x2(__uint_as_float(a[8 * q + 2]) * f, __uint_as_float(a[8 * q + 3]) * f),
                                  pack_bf16x2(__uint_as_float(a[8 * q + 4]) * f, __uint_as_float(a[8 * q + 5]) * f),
                                  pack_bf16x2(__uint_as_float(a[8 * q + 6]) * f, __uint_as_float(a[8 * q + 7]) * f));
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
gla_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                  const __grid_constant__ CUtensorMap tmDV, const BwdParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int dk = P.dkk, dv = P.dvv, H = P.H;
    const int nka = dk / 32, nva = dv / 64;
    const int slot = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant; which half of the work
    const int r = 32 * quad + lane;              // this thread's row (TMEM lane)

    const float ld = __ldg(P.log_decay + h);
    if (!(ld >= kFactoredMinLogDecay)) return;  // strong decay: the SIMT backward owns this head

    // (sequence, chunk) of this slot: the last sequence s with start_s / 128 + s <= slot
    int lo = 0, hi = P.nseq - 1, s = -1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int64_t st = P.cu ? (int64_t)__ldg(P.cu + mid) : (int64_t)mid * P.T;
        if (st / kC + mid <= slot) {
            s = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    if (s < 0) return;
    const int64_t start = P.cu ? (int64_t)__ldg(P.cu + s) : (int64_t)s * P.T;
    const int64_t len = P.cu ? (int64_t)__ldg(P.cu + s + 1) - start : (int64_t)P.T;
    if (len < 0) {
        if (tid == 0) record_status(GLA_ERR_DEVICE_ARG);
        return;
    }
    const int64_t c = (int64_t)slot - (start / kC + s);
    if (c * kC >= len) return;  // a slot past this sequence's chunks
    const int L = (int)((len - c * kC) < kC ? (len - c * kC) : kC);
    const int64_t row0 = start + c * kC;

    const BwdSmem plan = bwd_plan(dk, dv);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + plan.bars;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    float *tab = reinterpret_cast<float *>(smem + plan.tab);    // lambda^n, n = 0..128
    float *utab = reinterpret_cast<float *>(smem + plan.utab);  // lambda^-(j+1)
    float *wcol = reinterpret_cast<float *>(smem + plan.wcol);  // lambda^(i+1-L)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + plan.abort);
    const uint32_t tcols = kTmemCols;

    const int64_t img = ((int64_t)slot * H + h) * dk * dv;
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(BAR(B_LOAD), 1);
        mbar_init(BAR(B_LOAD2), 1);
        mbar_init(BAR(B_LOAD3), 1);
        mbar_init(BAR(B_MMA), 1);
        mbar_init(BAR(B_MASK), kThreads / 32);
        mbar_init(BAR(B_FINAL), 1);
        fence_mbar_init();
        // ---- loads, issued before the tables and the TMEM allocation so that those overlap the load
        // latency (a CTA handles one chunk: its prologue is not amortised) ----
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
        const uint32_t st_bytes = (uint32_t)dk * dv * 2u;
        const int y = (int)row0;
        mbar_expect_tx(BAR(B_LOAD), 2u * nka * 8192u);
        for (int a = 0; a < nka; ++a) {
            tma_load_2d(sb + plan.q + a * 8192u, &tmQ, h * dk + 32 * a, y, BAR(B_LOAD));
            tma_load_2d(sb + plan.k + a * 8192u, &tmK, h * dk + 32 * a, y, BAR(B_LOAD));
        }
        mbar_expect_tx(BAR(B_LOAD2), 2u * nva * 16384u + st_bytes);
        for (int a = 0; a < nva; ++a) {
            tma_load_2d(sb + plan.v + a * 16384u, &tmV, h * dv + 64 * a, y, BAR(B_LOAD2));
            tma_load_2d(sb + plan.dout + a * 16384u, &tmDO, h * dv + 64 * a, y, BAR(B_LOAD2));
        }
        bulk_load_g2s(sb + plan.g, P.g_img + img, st_bytes, BAR(B_LOAD2));
        mbar_expect_tx(BAR(B_LOAD3), st_bytes);
        bulk_load_g2s(sb + plan.s, P.s_img + img, st_bytes, BAR(B_LOAD3));
        tma_prefetch_desc(&tmDQ);
        tma_prefetch_desc(&tmDK);
        tma_prefetch_desc(&tmDV);
    }
    if (tid <= kC) tab[tid] = expf((float)tid * ld);
    if (tid < kC) utab[tid] = expf(-(float)(tid + 1) * ld);
    if (warp == 0) {
        tmem_alloc(sb + plan.slot, tcols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<uint32_t *>(smem + plan.slot);
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const uint32_t colDV = 0, colDK = (uint32_t)dv, colDQ = (uint32_t)(dv + dk);

    // descriptors
    const uint32_t qb = sb + plan.q, kb = sb + plan.k, vb = sb + plan.v, ob = sb + plan.dout;
    const uint32_t sI = sb + plan.s, gI = sb + plan.g;
    auto kmaj64 = [&](uint32_t base, int kk) {  // [128 x dk] tile, K-major over dk, 64B swizzle
        return smem_desc(base + (uint32_t)(kk >> 1) * 8192u + (uint32_t)(kk & 1) * 32u, 16, 512, kSwizzle64B);
    };
    auto mnmaj64 = [&](uint32_t base, int kk) {  // [128 x dk] tile read MN-major (MN = dk, K = tokens)
        return smem_desc(base + (uint32_t)kk * 1024u, 8192, 512, kSwizzle64B);
    };
    auto kmaj128 = [&](uint32_t base, uint32_t atom, int kk) {  // rows x dv, K-major over dv, 128B swizzle
        return smem_desc(base + (uint32_t)(kk >> 2) * atom + (uint32_t)(kk & 3) * 32u, 16, 1024, kSwizzle128B);
    };
    auto mnmaj128 = [&](uint32_t base, uint32_t atom, int kk) {  // MN = dv, K = rows (16 per step)
        return smem_desc(base + (uint32_t)kk * 2048u, atom, 1024, kSwizzle128B);
    };
    const uint32_t id_tt = idesc_bf16(kC, kC, 0, 0);    // 128 x 128 scores, both K-major
    const uint32_t id_pv = idesc_bf16(kC, dv, 0, 1);    // P (TMEM) x [tokens x dv] MN-major -> N = dv
    const uint32_t id_kg = idesc_bf16(kC, dv, 0, 1);    // K (K-major over dk) x G image (MN-major, N = dv)
    const uint32_t id_pq = idesc_bf16(kC, dk, 0, 1);    // P (TMEM) x [tokens x dk] MN-major -> N = dk
    const uint32_t id_vg = idesc_bf16(kC, dk, 0, 0);    // [tokens x dv] (K-major) x image^T (K-major, N = dk)
    const uint32_t vatom = 16384u, iatom = (uint32_t)dk * 128u;

    bool ok = true;
    // only the MMA issuer waits for loads; a failed wait sets the abort flag, which ends every other
    // wait of this CTA at once
    auto wait_load = [&](int b) {
        ok = ok && mbar_wait(BAR(b), 0, abort_flag, kWaitBudgetNs);
        if (!ok) *abort_flag = 1;
    };
    if (tid == 0) wait_load(B_LOAD);
    // ---- MMA1: A^T = K Q^T ----
    if (ok && tid == 0) {
        for (int kk = 0; kk < dk / 16; ++kk) mma_ss(tmem + kColScratch, kmaj64(kb, kk), kmaj64(qb, kk), id_tt, kk > 0);
        mma_commit(BAR(B_MMA));
    }
    // column factors of the dV / dK masks: lambda^(i+1-L); of the dQ mask: lambda^-(j+1) (utab)
    if (tid < kC) wcol[tid] = tab[min(tid + 1, kC)] * utab[max(L - 1, 0)];
    __syncthreads();

    int mma_phase = 0, mask_phase = 0;
    auto wait_mma = [&]() {
        ok = ok && mbar_wait(BAR(B_MMA), mma_phase & 1, abort_flag, kWaitBudgetNs);
        if (!ok) *abort_flag = 1;
        ++mma_phase;
        tc_fence_after();
    };
    auto masked = [&](bool lower, uint32_t colf) {
        // TMEM loads and stores are warp-collective: a warp takes part only if all its lanes are fine
        mask_scores(tmem + lane_base + kColScratch, r, L, lower, colf, half, __all_sync(0xffffffffu, ok) != 0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_MASK));
    };
    auto wait_mask = [&]() {  // thread 0 only
        ok = ok && mbar_wait(BAR(B_MASK), mask_phase & 1, abort_flag, kWaitBudgetNs);
        if (!ok) *abort_flag = 1;
        ++mask_phase;
        tc_fence_after();
    };

    // P1 = (A^T)_ji kept for i >= j, times lambda^(i+1-L)
    wait_mma();
    masked(false, sb + plan.wcol);
    if (tid == 0) {
        wait_mask();
        wait_load(B_LOAD2);
        if (ok) {
            // MMA2: dV = P1 dO + K G_c
            for (int kk = 0; kk < kC / 16; ++kk)
                mma_ts(tmem + colDV, tmem + kColScratch + (uint32_t)kk * 8u, mnmaj128(ob, vatom, kk), id_pv, kk > 0);
            for (int kk = 0; kk < dk / 16; ++kk) mma_ss(tmem + colDV, kmaj64(kb, kk), mnmaj128(gI, iatom, kk), id_kg, 1);
            // MMA3: B^T = V dO^T
            for (int kk = 0; kk < dv / 16; ++kk)
                mma_ss(tmem + kColScratch, kmaj128(vb, vatom, kk), kmaj128(ob, vatom, kk), id_tt, kk > 0);
            mma_commit(BAR(B_MMA));
        }
    }
    // P2 = (B^T)_ji kept for i >= j, times lambda^(i+1-L)
    wait_mma();
    masked(false, sb + plan.wcol);
    if (tid == 0) {
        wait_mask();
        if (ok) {
            // MMA4: dK = P2 Q + V G_c^T
            for (int kk = 0; kk < kC / 16; ++kk)
                mma_ts(tmem + colDK, tmem + kColScratch + (uint32_t)kk * 8u, mnmaj64(qb, kk), id_pq, kk > 0);
            for (int kk = 0; kk < dv / 16; ++kk) mma_ss(tmem + colDK, kmaj128(vb, vatom, kk), kmaj128(gI, iatom, kk), id_vg, 1);
            // MMA5: B = dO V^T
            for (int kk = 0; kk < dv / 16; ++kk)
                mma_ss(tmem + kColScratch, kmaj128(ob, vatom, kk), kmaj128(vb, vatom, kk), id_tt, kk > 0);
            mma_commit(BAR(B_MMA));
        }
    }
    // P3 = B_ij kept for j <= i, times lambda^-(j+1)
    wait_mma();  // MMA4, MMA5 done: dV and dK are final, and no MMA reads Q, V or G any more
    // A full chunk stages dV (over V) and dK (over Q) and starts their stores while mask 3 and MMA6 run,
    // so that only dQ is left once MMA6 is done.  One decision for the whole CTA (it has barriers).
    const bool early = __syncthreads_and(ok && L == kC) != 0;
    masked(true, sb + plan.utab);
    if (tid == 0) {
        wait_mask();
        wait_load(B_LOAD3);
        if (ok) {
            // MMA6: dQ = P3 K + dO S_{c-1}^T
            for (int kk = 0; kk < kC / 16; ++kk)
                mma_ts(tmem + colDQ, tmem + kColScratch + (uint32_t)kk * 8u, mnmaj64(kb, kk), id_pq, kk > 0);
            for (int kk = 0; kk < dv / 16; ++kk) mma_ss(tmem + colDQ, kmaj128(ob, vatom, kk), kmaj128(sI, iatom, kk), id_vg, 1);
            mma_commit(BAR(B_MMA));
        }
    }
    const float rf = tab[max(L - 1 - r, 0)];  // lambda^(L-1-j) for dV and dK
    const float qf = tab[min(r + 1, kC)];     // lambda^(i+1) for dQ
    if (early) {
        // the two halves of the warps split the dv + dk columns: dV's first columns to one, the rest of dV
        // and dK to the other
        const int vsplit = min(dv, 32 * ((dv + dk) / 64));
        if (half == 0) {
            stage_row(tmem + lane_base + colDV, 0, vsplit, rf, r, vb, 64);
        } else {
            stage_row(tmem + lane_base + colDV, vsplit, dv, rf, r, vb, 64);
            stage_row(tmem + lane_base + colDK, 0, dk, rf, r, qb, 32);
        }
        fence_async_shared();
        named_bar_sync(2, kThreads);
        if (tid == 0) {
            const int y = (int)row0;
            for (int a = 0; a < nva; ++a) tma_store_2d(&tmDV, h * dv + 64 * a, y, vb + a * 16384u);
            for (int a = 0; a < nka; ++a) tma_store_2d(&tmDK, h * dk + 32 * a, y, qb + a * 8192u);
            bulk_commit();
        }
    }
    wait_mma();

    // ---- epilogue: dQ (and for a partial chunk everything): row factors, bf16, rows below L ----
    ok = __syncthreads_and(ok) != 0;  // one decision for the whole CTA: the epilogue has a barrier
    if (ok) {
        if (L == kC) {
            // a full chunk (so `early` held): dQ staged over K, which MMA6 was the last to read, its 32-column
            // atoms split between the halves, and written with one store per atom
            const int qsplit = 32 * ((nka + 1) / 2);
            stage_row(tmem + lane_base + colDQ, half == 0 ? 0 : qsplit, half == 0 ? qsplit : dk, qf, r,
                      kb, 32);
            fence_async_shared();
            named_bar_sync(2, kThreads);
            if (tid == 0) {
                const int y = (int)row0;
                for (int a = 0; a < nka; ++a) tma_store_2d(&tmDQ, h * dk + 32 * a, y, kb + a * 8192u);
                bulk_commit();
            }
        } else {
            // the last chunk of a sequence: rows from L on belong to the next one; plain stores
            const bool live = r < L;
            const int64_t row = row0 + (r < L ? r : 0);
            if (half == 0) {
                store_row(tmem + lane_base + colDV, dv, rf, live, P.dv + (row * H + h) * dv);
            } else {
                store_row(tmem + lane_base + colDK, dk, rf, live, P.dk + (row * H + h) * dk);
                store_row(tmem + lane_base + colDQ, dk, qf, live, P.dq + (row * H + h) * dk);
            }
        }
    } else if (tid == 0) {
        record_status(GLA_ERR_TIMEOUT);
    }
    // the stores must have read shared memory before the CTA exits (also those of dV and dK when a later
    // wait gave up)
    if (tid == 0 && early) bulk_wait_read0();
    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        if (*abort_flag) {
            if (lane == 0) mma_commit(BAR(B_FINAL));
            __syncwarp();
            mbar_wait(BAR(B_FINAL), 0, nullptr, kWaitBudgetNs);
        }
        tmem_dealloc(tmem, tcols);
    }
#undef BAR
}

}  // namespace

bool tc_bwd_supported(int dk, int dv, int chunk) {
    if (!tc_chunk_supported(dk, dv, chunk)) return false;  // the state passes run on the forward kernel
    if (!(chunk == kC && dk % 32 == 0 && dk >= 32 && dk <= 128 && dv % 64 == 0 && dv >= 64 && dv <= 192 &&
          dv + 2 * dk <= (int)kColScratch))
        return false;
    return bwd_plan(dk, dv).total + 1024 <= (uint32_t)device_info().max_smem_optin;
}

// Backward on the tensor cores: two state passes, the chunk-parallel gradient kernel, then the
// chunked SIMT backward for the heads whose decay is too strong for the factored masks (its CTAs
// return at once for every other head).  Scratch: two bf16 state tiles per chunk slot.
// With `s_images` non-null (the states before every chunk, left by the forward) the forward state pass
// is skipped and only the gradient-state images are scratch.
// A non-blocking stream per device for work forked off the caller's stream and joined back to it
// before the call returns (created once; null if that failed).
cudaStream_t side_stream() {
    constexpr int kMaxDev = 64;
    static std::once_flag once[kMaxDev];
    static cudaStream_t streams[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::call_once(once[dev], [dev]() {
        if (cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            streams[dev] = nullptr;
        }
    });
    return streams[dev];
}

static int chunk_bwd_impl(const void *q, const void *k, const void *v, const void *dout, const float *ld, const float *h0,
                   const float *dhT, const void *s_images, void *dq, void *dk_, void *dv_, float *dh0, int nseq,
                   int Tlen, int H, int dk, int dv, const int32_t *cu, cudaStream_t st) {
    if (!tc_bwd_supported(dk, dv, kC)) return GLA_ERR_UNSUPPORTED;
    const uint64_t rows = cu ? (uint64_t)Tlen : (uint64_t)nseq * (uint64_t)Tlen;
    if (rows >= (1ull << 31)) return GLA_ERR_UNSUPPORTED;
    const long long slots = (long long)(rows / kC) + nseq + 1;
    if (slots * H > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv, mo, mdq, mdk, mdv;
    if (!make_map(&mq, q, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B, kC) ||
        !make_map(&mk, k, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B, kC) ||
        !make_map(&mv, v, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B, kC) ||
        !make_map(&mo, dout, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B, kC) ||
        !make_map(&mdq, dq, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B, kC) ||
        !make_map(&mdk, dk_, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B, kC) ||
        !make_map(&mdv, dv_, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B, kC))
        return GLA_ERR_LAUNCH;
    const size_t per = (size_t)slots * H * dk * dv;  // bf16 elements per image array
    const size_t nimg = s_images ? 1 : 2;
    __nv_bfloat16 *img = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&img), nimg * per * sizeof(__nv_bfloat16), st) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_NOMEM;
    }
    const __nv_bfloat16 *s_img = s_images ? reinterpret_cast<const __nv_bfloat16 *>(s_images) : img;
    __nv_bfloat16 *g_img = img + (nimg - 1) * per;
    // The chunked SIMT recurrences own the heads with strong decays (their CTAs of other heads return at
    // once); they touch other heads' gradients than the tensor-core kernels, so they run on a side
    // stream forked here and joined at the end instead of adding three launches to this stream.
    cudaStream_t side = side_stream();
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
    bool forked = false;
    if (side && cudaEventCreateWithFlags(&fork_ev, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventCreateWithFlags(&join_ev, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventRecord(fork_ev, st) == cudaSuccess && cudaStreamWaitEvent(side, fork_ev, 0) == cudaSuccess)
        forked = true;
    else
        cudaGetLastError();
    int rc_strong = GLA_OK;
    if (forked) {
        rc_strong = simt_chunk_bwd_bf16_strong(q, k, v, dout, ld, h0, dhT, dq, dk_, dv_, dh0, nseq, Tlen, H, dk, dv,
                                               kC, cu, side);
        if (cudaEventRecord(join_ev, side) != cudaSuccess) rc_strong = GLA_ERR_LAUNCH;
    }
    int rc = s_images ? GLA_OK : tc_state_pass_bf16(k, v, ld, h0, nullptr, img, 0, nseq, Tlen, H, dk, dv, cu, st);
    if (rc == GLA_OK) rc = tc_state_pass_bf16(q, dout, ld, dhT, dh0, g_img, 1, nseq, Tlen, H, dk, dv, cu, st);
    if (rc == GLA_OK) {
        const size_t bytes = bwd_plan(dk, dv).total + 1024;
        if (cudaFuncSetAttribute(gla_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
            cudaSuccess) {
            rc = GLA_ERR_LAUNCH;
        } else {
            BwdParams p{};
            p.log_decay = ld;
            p.cu = cu;
            p.s_img = s_img;
            p.g_img = g_img;
            p.dq = reinterpret_cast<__nv_bfloat16 *>(dq);
            p.dk = reinterpret_cast<__nv_bfloat16 *>(dk_);
            p.dv = reinterpret_cast<__nv_bfloat16 *>(dv_);
            p.nseq = nseq;
            p.T = Tlen;
            p.H = H;
            p.dkk = dk;
            p.dvv = dv;
            p.slots = (int)slots;
            gla_bwd_tc_kernel<<<(unsigned)(slots * H), kThreads, bytes, st>>>(mq, mk, mv, mo, mdq, mdk, mdv, p);
            count_launches(1);
            rc = cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
        }
    }
    if (forked) {
        if (cudaStreamWaitEvent(st, join_ev, 0) != cudaSuccess && rc == GLA_OK) rc = GLA_ERR_LAUNCH;
        if (rc == GLA_OK) rc = rc_strong;
    } else if (rc == GLA_OK) {
        rc = simt_chunk_bwd_bf16_strong(q, k, v, dout, ld, h0, dhT, dq, dk_, dv_, dh0, nseq, Tlen, H, dk, dv, kC, cu,
                                        st);
    }
    if (fork_ev) cudaEventDestroy(fork_ev);
    if (join_ev) cudaEventDestroy(join_ev);
    cudaFreeAsync(img, st);
    return rc;
}

int tc_chunk_bwd_bf16(const void *q, const void *k, const void *v, const void *dout, const float *ld,
                      const float *h0, const float *dhT, void *dq, void *dk_, void *dv_, float *dh0, int nseq,
                      int Tlen, int H, int dk, int dv, const int32_t *cu, cudaStream_t st) {
    return chunk_bwd_impl(q, k, v, dout, ld, h0, dhT, nullptr, dq, dk_, dv_, dh0, nseq, Tlen, H, dk, dv, cu, st);
}

int tc_chunk_bwd_bf16_saved(const void *q, const void *k, const void *v, const void *dout, const float *ld,
                            const float *h0, const float *dhT, const void *s_images, void *dq, void *dk_, void *dv_,
                            float *dh0, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu, cudaStream_t st) {
    return chunk_bwd_impl(q, k, v, dout, ld, h0, dhT, s_images, dq, dk_, dv_, dh0, nseq, Tlen, H, dk, dv, cu, st);
}

}  // namespace gla
