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
// four contractions are tcgen05.mma instructions (M = 128, K-steps of 16), issued
// in the order MMA1, MMA3, MMA2, MMA4 by the passes that write outputs (the
// state-only passes run MMA4 alone):
//   MMA1  A    = Q K^T                      TMEM cols [384, 512)   A: Q (smem), B: K (smem)
//   MMA3  O    = (diag(lambda^(i+1)) Q) S   TMEM cols [0, dv)      A: Q' (smem), B: S bf16 (smem)
//   MMA4  S   += (diag(lambda^(L-1-j)) K)^T V  TMEM cols [192, 192+dv)  A: K'^T (smem), B: V (smem)
//   MMA2  O   += P V,  P = bf16(A .* D)     A: P (TMEM, aliases A), B: V (smem)
// The state rows are dk (<= 128), padded to M = 128; rows >= dk of the state
// accumulator are never read.
//
// Warp roles (448 threads):
//   warps 0-3  "state" warpgroup: thread t owns TMEM lane t (a dk row of S).
//              Per chunk: state pass (read the state accumulator from TMEM,
//              finish S_{c-1}, write its bf16 copy for MMA3 and the f32 value
//              back for MMA4), then the K row decays in place (and, for strong
//              decays, the Q row decays).
//   warps 4-7  "mask" warpgroup: thread t owns TMEM lane t - 128 (a token row).
//              Per chunk: mask A -> P.
//   warps 10-13 "epilogue" warpgroup (TMEM lane quadrant = warp % 4): O (TMEM)
//              -> bf16, 64 columns at a time, into a 4 KB staging tile per
//              warp laid out as a 128B-swizzled TMA box, then one TMA store
//              per tile; a tile is refilled once its previous store has read
//              it.  O leaves TMEM at the pace of the TMEM loads, so MMA3 of
//              the next chunk is not held up by global stores.  The mask of
//              chunk c+1 and the epilogue of chunk c overlap.  (Gated instance:
//              O times the output gate's factor, see the gated loop below.)
//   warp 8     TMA producer.  Passes that write outputs: Q and K and V double
//              buffered with a barrier pair per tile (Q(c+2) once MMA3(c) is
//              done, K(c+2) once MMA4(c) is, V(c+1) once MMA3(c) has read the
//              state copy in its tile); state-only passes: K/V stages.
//   warp 9     MMA issuer and TMEM owner.
//   One count-8 barrier (SREADY) lets MMA3 go: the state warps' copy of
//   S_{c-1} and the epilogue warps' release of O.
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
//                (dk rows x 128 B).  MN-major B operand of MMA3.  In the passes
//                that write outputs it is written into the V tile of the
//                previous chunk (smem_plan_full); in the others it has a tile
//                of its own (smem_plan).
#include <atomic>
#include <mutex>

#include "gla_common.cuh"
#include "sm100_ptx.cuh"

GLA_DEFINE_STATUS(tc)

namespace gla {
namespace {

using namespace ptx;

constexpr int kC = 128;              // chunk length (MMA M and the token K extent)
constexpr int kThreads = 448;        // state, mask and epilogue warpgroups + producer + MMA warp
constexpr int kEpiWarp0 = 10;        // first warp of the epilogue warpgroup
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;        // O accumulator  [0, dv)
constexpr uint32_t kColS = 192;      // state          [192, 192 + dv)
constexpr uint32_t kColA = 384;      // A = Q K^T      [384, 512); P aliases [384, 448)
constexpr uint64_t kWaitBudgetNs = 4000000000ull;  // 4 s per wait

// Launch modes.  A long dense sequence with few (sequence, head) chains is cut into nseg
// segments of seg_chunks chunks: pass 1 (kStateOnly) computes every segment's end state from a zero
// start, a small scan turns those into the segment start states, and pass 2 (kSegmented) runs the
// full forward of every segment from its start state.
//
// kStates is the state pass of the backward: a state-only walk over whole chains, forwards or
// backwards in time, that also writes the state in force before every chunk (the bf16 tile MMA3
// would read, as a raw shared-memory image) to chunk_states.  Forwards it gives the S_{c-1} of the
// chunks from h0; backwards, with the tiles of q and dout in the roles of k and v, it gives the
// gradient states G_c = dL/dS_c from dhT:  G_{c-1} = lambda^L G_c + sum_i lambda^(i+1) q_i^T do_i,
// and dh0 as its final state.
enum Mode : int { kWhole = 0, kStateOnly = 1, kSegmented = 2, kStates = 3 };

struct Params {
    const float *log_decay;
    const float *h0;       // [nseq, H, dk, dv] or null
    __nv_bfloat16 *out;
    float *hT;             // [nseq, H, dk, dv] or null
    const int32_t *cu;
    int T, H, dk, dv;
    int mode;              // Mode
    int nseg;              // segments per chain (1 for kWhole)
    int seg_chunks;        // chunks per segment (segmented modes)
    int grid_seg;          // segments per chain in this launch (nseg - 1 for kStateOnly)
    const float *seg_h0;   // kSegmented: start states of segments 1..nseg-1, [chains, nseg-1, dk, dv]
    float *seg_end;        // kStateOnly: end states of segments 0..nseg-2 from zero, [chains, nseg-1, dk, dv]
    int reverse;           // kStates: walk the chunks backwards in time (launches the kRev kernel)
    __nv_bfloat16 *chunk_states;  // kStates: [slots, H, dk*dv] state images; chunk c of sequence s at
                                  // slot start_s / 128 + s + c (start_s its first row)
    int nseq;              // sequences (packed batches: entries of cu minus one)
    int lpt;               // packed batch, whole chains: CTA i takes the sequence of length rank i / H
    const __nv_bfloat16 *gate;  // full passes with the output gate: [rows, H, dv] like out (kGate instance)
    int gate_kind;              // 0: out = O * SiLU(g); 1: out = O * sigmoid(g)
};

// Packed batches of up to this many sequences are walked longest first (the ranking costs every CTA
// O(nseq^2 / threads) comparisons in its prologue).
constexpr int kLptMaxSeq = 256;

// Shared memory plan (bytes from the 1024-aligned base).
struct Smem {
    uint32_t q, q1, k0, k1, v0, v1, s, gb, xp, tab, utab, bars, slot, abort, total;
};

// Barriers, lookup tables and the TMEM slot after the tiles at offset `at`.
__host__ __device__ constexpr void smem_plan_tail(Smem &p, uint32_t at) {
    p.xp = at;                   // output staging: 4 warps x 32 rows x 128 B
    p.tab = p.xp + 4u * 4096u;
    p.utab = p.tab + 132 * 4;
    p.bars = p.utab + 128 * 4;
    p.bars = (p.bars + 7u) & ~7u;
    p.slot = p.bars + 40 * 8;  // room for up to 40 barriers
    p.abort = p.slot + 4;
    p.total = p.abort + 4;
}

__host__ __device__ constexpr Smem smem_plan(int dk, int dv) {
    Smem p{};
    const uint32_t qk = (uint32_t)(dk / 32) * 8192u;
    const uint32_t vv = (uint32_t)(dv / 64) * 16384u;
    p.q = 0;
    p.q1 = p.q;
    p.k0 = p.q + qk;
    p.k1 = p.k0 + qk;
    p.v0 = p.k1 + qk;  // MMA4 reads up to 4 atoms from a K tile: V follows, so the over-read stays in bounds
    p.v1 = p.v0 + vv;
    p.s = p.v1 + vv;
    p.gb = 0;
    smem_plan_tail(p, p.s + (uint32_t)dk * 128u * (uint32_t)(dv / 64));
    return p;
}

// The full passes (outputs and states): two Q tiles, so that the next chunk's Q is in flight while the
// current one is still read, and no state-copy tile of its own.  The bf16 copy of S_{c-1} that MMA3(c)
// reads is written into the V tile of chunk c-1 (free once MMA2(c-1) and MMA4(c-1) are done; dk <= 128
// rows of dv bf16 fit in its 128 rows), and V(c+1) lands there once MMA3(c) has read it.
__host__ __device__ constexpr Smem smem_plan_full(int dk, int dv, bool gate = false) {
    Smem p{};
    const uint32_t qk = (uint32_t)(dk / 32) * 8192u;
    const uint32_t vv = (uint32_t)(dv / 64) * 16384u;
    p.q = 0;
    p.q1 = p.q + qk;
    p.k0 = p.q1 + qk;
    p.k1 = p.k0 + qk;
    p.v0 = p.k1 + qk;  // as above: the over-read of K1 by MMA4 stays inside V0
    p.v1 = p.v0 + vv;
    p.s = p.v0;        // no tile of its own (see above)
    p.gb = p.v1 + vv;  // gated instance: 4 x 4 KB of output-gate rows (one 64-column group per epilogue warp)
    smem_plan_tail(p, p.gb + (gate ? 4u * 4096u : 0u));
    return p;
}

// barrier indices
// Every barrier that can be arrived on for chunk c+1 before its waiter has passed chunk c is kept per
// K/V stage (KPREP: the K rows of chunk c+1 may be ready before the MMA warp has waited for chunk c's);
// with parity waits, a barrier must never run two phases ahead of a waiter.
// In the full passes the K/V barriers of a stage track the K tile alone, and the V tile and the second Q
// tile have barriers of their own.
enum { B_QFULL = 0, B_QEMPTY, B_KVFULL0, B_KVFULL1, B_KVEMPTY0, B_KVEMPTY1, B_AFULL, B_KPREP0, B_KPREP1, B_SREADY,
       B_PFULL, B_OFULL, B_SFULL, B_FINAL, B_KVFULL2, B_KVEMPTY2, B_KPREP2, B_IMGDONE,
       B_QFULL1, B_QEMPTY1, B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1, B_COUNT };
// barrier of K/V stage s (a state-only pass runs three stages, every other pass two)
__device__ __forceinline__ int b_kvfull(int s) { return s == 0 ? B_KVFULL0 : s == 1 ? B_KVFULL1 : B_KVFULL2; }
__device__ __forceinline__ int b_kvempty(int s) { return s == 0 ? B_KVEMPTY0 : s == 1 ? B_KVEMPTY1 : B_KVEMPTY2; }
__device__ __forceinline__ int b_kprep(int s) { return s == 0 ? B_KPREP0 : s == 1 ? B_KPREP1 : B_KPREP2; }
// the gated instance's epilogue warps add two gate barriers each after B_COUNT
static_assert(B_COUNT + 8 <= 40, "the shared-memory plan reserves 40 barrier slots");

// Output-gate factors in the tensor-core epilogue, which drains O on the chunk loop's critical path: two
// gate values at a time in bf16 pairs, sigmoid(g) = (1 + tanh(g/2)) / 2 and SiLU(g) = g sigmoid(g) with the
// hardware tanh approximation (one MUFU operation per pair).  The factors carry bf16 precision and an
// absolute sigmoid error of a few 1e-3 at most, about the bf16 rounding of the output itself; the drain
// multiplies them by the row factor and by O rounded to bf16 in bf16 pairs as well.
__device__ __forceinline__ uint32_t gate_factor_bf16x2(uint32_t g2, int kind) {
    const uint32_t half2 = 0x3f003f00u;  // (0.5, 0.5) in bf16
    uint32_t hg, t, f;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hg) : "r"(g2), "r"(half2));
    asm("tanh.approx.bf16x2 %0, %1;" : "=r"(t) : "r"(hg));
    if (kind == 0)
        asm("fma.rn.bf16x2 %0, %1, %2, %1;" : "=r"(f) : "r"(hg), "r"(t));  // hg t + hg
    else
        asm("fma.rn.bf16x2 %0, %1, %2, %2;" : "=r"(f) : "r"(t), "r"(half2));  // t / 2 + 1 / 2
    return f;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Two f32 values (bit patterns) times the pair g2 with one instruction: mul.rn.f32x2 rounds each lane as
// mul.rn.f32 does, so the results are those of two scalar multiplies.
__device__ __forceinline__ uint64_t f32x2_splat(float g) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(g));
    return d;
}
__device__ __forceinline__ void mul_f32x2(uint32_t &lo, uint32_t &hi, uint64_t g2) {
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%0, %1};\n\tmul.rn.f32x2 t, t, %2;\n\tmov.b64 {%0, %1}, t;\n\t}"
        : "+r"(lo), "+r"(hi)
        : "l"(g2));
}
// 32 values in place, in pairs
__device__ __forceinline__ void scale32(uint32_t (&v)[32], uint64_t g2) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) mul_f32x2(v[e], v[e + 1], g2);
}

// The four contractions as groups of K-steps of 16, fully unrolled, with every operand descriptor advanced
// by a constant from a base computed once: the MMA warp spends a few instructions per tcgen05.mma, so the
// tensor pipe is not left waiting for it to issue.  A descriptor holds its start address in 16-byte units,
// so a byte offset o adds o >> 4 (shared-memory offsets stay below 256 KB: no carry out of the field).
// Q, K tiles (K-major, 64B swizzle): K-step kk is 32 bytes into atom kk / 2 (8 KB apart).
__device__ __forceinline__ uint64_t qk_step(int kk) { return (uint64_t)((kk >> 1) * 512 + (kk & 1) * 2); }

// MMA1: A = Q K^T (ksteps = dk / 16 <= 8), both operands K-major.
__device__ __forceinline__ void mma_group_qk(uint32_t d, uint64_t dq, uint64_t dk_, uint32_t id, int ksteps) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        if (kk < ksteps) mma_ss(d, dq + qk_step(kk), dk_ + qk_step(kk), id, kk > 0);
}
// MMA3: O = Q S; B = the bf16 state copy, MN-major, 2 KB per K-step of 16 dk rows.
__device__ __forceinline__ void mma_group_qs(uint32_t d, uint64_t dq, uint64_t ds, uint32_t id, int ksteps) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        if (kk < ksteps) mma_ss(d, dq + qk_step(kk), ds + (uint64_t)(kk * 128), id, kk > 0);
}
// MMA2: O += P V; A = P in TMEM (8 columns per K-step of 16 tokens), B = V MN-major (2 KB per K-step).
__device__ __forceinline__ void mma_group_pv(uint32_t d, uint32_t p_tmem, uint64_t dv_, uint32_t id) {
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) mma_ts(d, p_tmem + (uint32_t)(kk * 8), dv_ + (uint64_t)(kk * 128), id, 1);
}
// MMA4: S += K~^T V; A = K tile read MN-major (1 KB per K-step of 16 tokens), B = V MN-major.
__device__ __forceinline__ void mma_group_kv(uint32_t d, uint64_t dkt, uint64_t dv_, uint32_t id) {
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) mma_ss(d, dkt + (uint64_t)(kk * 64), dv_ + (uint64_t)(kk * 128), id, 1);
}
// Base descriptors of the operand roles.
__device__ __forceinline__ uint64_t desc_qk(uint32_t a) { return smem_desc(a, 16, 512, kSwizzle64B); }
__device__ __forceinline__ uint64_t desc_kt(uint32_t a) { return smem_desc(a, 8192, 512, kSwizzle64B); }
__device__ __forceinline__ uint64_t desc_v(uint32_t a) { return smem_desc(a, 16384, 1024, kSwizzle128B); }
__device__ __forceinline__ uint64_t desc_s(uint32_t a, int dk) { return smem_desc(a, (uint32_t)dk * 128u, 1024, kSwizzle128B); }

// Multiply the 16-byte chunk at `p` (8 bf16) by f, in place.
__device__ __forceinline__ void scale_chunk_bf16(uint8_t *p, uint64_t f2) {
    uint4 x = *reinterpret_cast<uint4 *>(p);
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        uint32_t lo = w[e] << 16, hi = w[e] & 0xffff0000u;  // the bf16 pair as two f32 values
        mul_f32x2(lo, hi, f2);
        w[e] = pack_bf16x2(__uint_as_float(lo), __uint_as_float(hi));
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Scale row r of a [128 x dk] tile stored as 64B-swizzled atoms (8 KB each).  The
// swizzle only permutes the four 16-byte chunks inside a row, and every chunk gets
// the same factor, so the row is walked in the order that spreads a warp's 32 rows
// over all banks: chunk i of thread r is physical chunk i ^ ((r >> 1) & 3).
__device__ __forceinline__ void scale_row_sw64(uint8_t *tile, int nka, int r, float f) {
    const int x = (r >> 1) & 3;
    const uint64_t f2 = f32x2_splat(f);
    for (int a = 0; a < nka; ++a) {
        uint8_t *row = tile + a * 8192 + r * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) scale_chunk_bf16(row + ((i ^ x) << 4), f2);
    }
}

// kRev: the reversed state pass of the backward (kStates with reverse set); a separate instantiation
// so that the forward's register allocation is untouched.  kNst: K/V stages in flight; the forward's
// state-only pass has three (its third K tile takes the unused Q buffer, its third V tile the unused
// state-copy and output-staging space), every other pass two.  kFull: the passes that compute outputs
// (kWhole, kSegmented), with the shared-memory plan of smem_plan_full; the other instances run the
// state-only modes.  kGate: a full pass that multiplies every output by the output gate's factor.
template <bool kRev, int kNst, bool kFull, bool kGate = false>
__global__ void __launch_bounds__(kThreads, 1)
gla_tc_chunk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmG, const Params P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 1024-aligned base, by pointer arithmetic on the shared array (not through an integer), so that
    // every access derived from it compiles to a shared-memory instruction
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int dk = P.dk, dv = P.dv, H = P.H;
    const int nka = dk / 32, nva = dv / 64;
    // shared-memory offsets (scalars: nothing of the plan lives in local memory)
    const Smem plan = kFull ? smem_plan_full(dk, dv, kGate) : smem_plan(dk, dv);
    const uint32_t o_q = plan.q, o_k0 = plan.k0, o_k1 = plan.k1, o_v0 = plan.v0, o_v1 = plan.v1, o_s = plan.s;
    const uint32_t o_q1 = plan.q1, o_gb = plan.gb;
    const uint32_t o_xp = plan.xp;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + plan.bars;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    float *tab = reinterpret_cast<float *>(smem + plan.tab);    // lambda^n,      n = 0..128
    float *utab = reinterpret_cast<float *>(smem + plan.utab);  // lambda^-(j+1), j = 0..127 (factored form)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + plan.slot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + plan.abort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool rev = kRev;
    // segment w in walk order of this CTA's chain; walked backwards in time, walk order runs from the
    // sequence's last segment to its first
    const int chain = blockIdx.x / P.grid_seg, w = blockIdx.x % P.grid_seg;
    const int seg = rev ? P.nseg - 1 - w : w;  // natural segment
    const int h = chain % H;
    int seq = chain / H;
    if (P.lpt) {
        // Longest sequences first: the CTAs of a packed batch start in blockIdx order as SMs free up, so a
        // long sequence late in the batch would trail the whole launch.  CTA i takes the sequence whose
        // length ranks i / H in decreasing order (ties by index: a permutation even for bad offsets, which
        // seq_range reports below).  The lengths sit in the output staging tiles, unused until the first
        // epilogue; the pick in the entry after them.
        int *lens = reinterpret_cast<int *>(smem + plan.xp);
        for (int s = threadIdx.x; s < P.nseq; s += blockDim.x) lens[s] = __ldg(P.cu + s + 1) - __ldg(P.cu + s);
        __syncthreads();
        const int want = chain / H;
        for (int s = threadIdx.x; s < P.nseq; s += blockDim.x) {
            const int ls = lens[s];
            int rank = 0;
            for (int u = 0; u < P.nseq; ++u) {
                const int lu = lens[u];
                rank += (lu > ls || (lu == ls && u < s)) ? 1 : 0;
            }
            if (rank == want) lens[P.nseq] = s;
        }
        __syncthreads();
        seq = lens[P.nseq];
    }
    const bool state_only = !kFull;
    const bool write_images = !kFull && P.mode == kStates && P.chunk_states != nullptr;
    // The full forward can also leave the state in force before every chunk, as the bf16 tile MMA3 reads,
    // in the layout the backward consumes (training: the backward then skips its forward state pass).
    const bool save_images = kFull && P.chunk_states != nullptr;
    const bool segmented = P.mode == kStateOnly || P.mode == kSegmented || (P.mode == kStates && P.nseg > 1);

    SeqRange rng;
    const bool valid = seq_range(seq, P.T, P.cu, rng);
    int64_t len = valid ? rng.len : 0;
    int64_t start = rng.start;
    if (segmented) {  // one segment of a dense sequence
        const int64_t s0 = (int64_t)seg * P.seg_chunks * kC;
        start += s0;
        len = (len - s0 < (int64_t)P.seg_chunks * kC) ? len - s0 : (int64_t)P.seg_chunks * kC;
    }
    const int nchunks = (int)((len + kC - 1) / kC);
    const int row0 = (int)start;
    // where the chain segment's initial state comes from and where its final state goes (null: zeros / none)
    const int64_t sz_state = (int64_t)P.dk * P.dv;
    const float *init_state = P.h0 ? P.h0 + ((int64_t)seq * H + h) * sz_state : nullptr;
    float *final_state = P.hT ? P.hT + ((int64_t)seq * H + h) * sz_state : nullptr;
    // per chain, segment scratch is [nseg - 1] states in walk order: the end states from zero of walk
    // segments 0..nseg-2 (pass 1), and the start states of walk segments 1..nseg-1 (after the scan)
    if (P.mode == kStateOnly) {
        init_state = nullptr;
        final_state = P.seg_end + ((int64_t)chain * (P.nseg - 1) + w) * sz_state;
    } else if (segmented) {
        if (w > 0) init_state = P.seg_h0 + ((int64_t)chain * (P.nseg - 1) + w - 1) * sz_state;
        if (w < P.nseg - 1) final_state = nullptr;
    }
    // The state warps read the initial state at their first state pass, a row per thread in 64-column
    // groups, one after the other; in a walk over a whole chain (h0 from DRAM) its lines are asked into
    // L2 here, before the barriers, tables and TMEM allocation, so that the later groups do not each wait
    // for DRAM (ragged batch of 1,024 chains: 776 -> 768 us).  Segment start states come from the scan,
    // which has just written them.
    if (!segmented && init_state != nullptr && (int)threadIdx.x < P.dk) {
        const char *row = reinterpret_cast<const char *>(init_state + (int64_t)threadIdx.x * P.dv);
        for (int o = 0; o < P.dv * 4; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + o));
    }
    const float ld = __ldg(P.log_decay + h);
    const float lam = expf(ld);
    // Factored decay: lambda^(i-j) = lambda^(i+1) * lambda^-(j+1).  K rows are scaled by lambda^-(j+1)
    // once (K''), which serves both A = Q K''^T (the decay mask becomes a plain causal mask) and the
    // state update S_c = lambda^L (S_{c-1} + K''^T V); the row factor lambda^(i+1) is applied to O in
    // the epilogue, so Q needs no rescaled copy.  Used while lambda^-128 stays far from overflow
    // (lambda >= e^-0.3); stronger decays take the direct form: Q rows scaled by lambda^(i+1), K rows
    // by lambda^(L-1-j), per-element decay in the mask, state pre-scaled by lambda^L.
    const bool fact = ld >= -0.3f;
    // The forward's state-only pass with a factored decay keeps the state in a frame that moves only
    // every nblk chunks: within a block the K rows of its m-th chunk carry lambda^-(m*128 + j + 1), so
    // the MMAs of consecutive chunks accumulate without a state pass between them, and at the block
    // end one pass scales the state by lambda^(rows of the block).  nblk keeps every frame factor
    // below e^36 (the latest rows, whose weight in the result is about 1, carry the largest).
    const bool blocked = !kFull && P.mode == kStateOnly && fact;
    // The backward's state passes (kStates) with a factored decay use the same moving frame; the
    // state before each chunk, for its image, is lambda^(rows walked in the block so far) times the
    // frame, so only the block ends write the state back to TMEM, and the image's copy out of shared
    // memory runs while the next MMA does.
    const bool framed = !kFull && P.mode == kStates && fact;
    // The backward does not use the state passes' results for strong decays (the chunked SIMT
    // recurrences own those heads, dh0 included), so their CTAs have nothing to do.
    if (!kFull && P.mode == kStates && !fact) return;
    int nblk = 1;
    if (blocked || framed) {
        const float a = -ld * (float)kC;  // >= 0
        nblk = (a > 0.f) ? (int)fminf(64.f, fmaxf(1.f, floorf(36.f / a))) : 64;
    }
    auto chunk_len = [&](int c) -> int {
        const int64_t rem = len - (int64_t)c * kC;
        return (int)(rem < kC ? rem : kC);
    };
    // the c-th chunk walked (backwards in time for a reversed state pass) and its length
    auto nat = [&](int c) -> int { return rev ? nchunks - 1 - c : c; };
    auto plen = [&](int c) -> int { return chunk_len(nat(c)); };
    auto stg = [&](int c) -> int { return c % kNst; };          // K/V stage of the c-th chunk walked
    auto sph = [&](int c) -> uint32_t { return (uint32_t)(c / kNst) & 1u; };  // its phase on that stage
    auto kbuf_of = [&](int s) -> uint32_t { return s == 0 ? o_k0 : s == 1 ? o_k1 : o_q; };
    auto vbuf_of = [&](int s) -> uint32_t { return s == 0 ? o_v0 : s == 1 ? o_v1 : o_s; };
    // full passes: Q tile of chunk c, and the state copy S_{c-1} that MMA3(c) reads (in V tile c-1; the
    // copy of h0 for chunk 0 in the V tile that chunk 1 takes)
    auto qbuf_of = [&](int c) -> uint32_t { return kFull ? ((c & 1) ? o_q1 : o_q) : o_q; };
    auto scopy_of = [&](int c) -> uint32_t { return kFull ? ((c & 1) ? o_v0 : o_v1) : o_s; };

    if (threadIdx.x == 0) {
        if (!valid) record_status(GLA_ERR_DEVICE_ARG);
        *abort_flag = 0;
        mbar_init(BAR(B_QFULL), 1);
        mbar_init(BAR(B_QEMPTY), 1);
        mbar_init(BAR(B_KVFULL0), 1);
        mbar_init(BAR(B_KVFULL1), 1);
        mbar_init(BAR(B_KVEMPTY0), 1);
        mbar_init(BAR(B_KVEMPTY1), 1);
        mbar_init(BAR(B_AFULL), 1);
        mbar_init(BAR(B_KPREP0), 4);
        mbar_init(BAR(B_KPREP1), 4);
        // full passes: the state warps' copy (and, direct form, Q prep) plus the epilogue warps' release
        // of O, so that MMA3 waits on one barrier
        mbar_init(BAR(B_SREADY), kFull ? 8 : 4);
        mbar_init(BAR(B_PFULL), 4);
        mbar_init(BAR(B_OFULL), 1);
        mbar_init(BAR(B_SFULL), 1);
        mbar_init(BAR(B_FINAL), 1);
        mbar_init(BAR(B_KVFULL2), 1);
        mbar_init(BAR(B_KVEMPTY2), 1);
        mbar_init(BAR(B_KPREP2), 4);
        mbar_init(BAR(B_IMGDONE), 1);
        mbar_init(BAR(B_QFULL1), 1);
        mbar_init(BAR(B_QEMPTY1), 1);
        mbar_init(BAR(B_VFULL0), 1);
        mbar_init(BAR(B_VFULL1), 1);
        // a V tile holds a state copy until MMA3 has read it, and, when images are saved, until the
        // image store has too
        mbar_init(BAR(B_VEMPTY0), save_images ? 2 : 1);
        mbar_init(BAR(B_VEMPTY1), save_images ? 2 : 1);
        if (kGate)  // gated drain: per epilogue warp, one barrier per gate buffer (TMA loads of 4 KB)
            for (int i = 0; i < 8; ++i) mbar_init(BAR(B_COUNT + i), 1);
        fence_mbar_init();
    }
    if (threadIdx.x < kC + 4) tab[threadIdx.x] = (threadIdx.x <= kC) ? expf((float)threadIdx.x * ld) : 0.f;
    if (threadIdx.x < kC) utab[threadIdx.x] = fact ? expf(-(float)(threadIdx.x + 1) * ld) : 0.f;
    if (warp == kMmaWarp) {
        tmem_alloc(sbase + plan.slot, kTmemCols);
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
            if (!state_only) tma_prefetch_desc(&tmO);
            if (kGate) tma_prefetch_desc(&tmG);
            const uint32_t kvbytes = (uint32_t)nka * 8192u + (uint32_t)nva * 16384u;
            const uint32_t qbytes = (uint32_t)nka * 8192u;
            bool ok = true;
            for (int c = 0; c < nchunks && ok && kFull; ++c) {
                // full passes: Q(c) into its tile once MMA3(c-2) is done, K(c) once MMA4(c-2) is, V(c) once
                // MMA3(c-1) has read the state copy in its tile (waits in issue order of their releases)
                const int s = c & 1;
                const int y = row0 + c * kC;
                const uint32_t nfree = (uint32_t)((c >> 1) - 1) & 1u;  // phase of the release by chunk c-2
                const int bqf = s ? B_QFULL1 : B_QFULL, bqe = s ? B_QEMPTY1 : B_QEMPTY;
                if (c >= 2 && !(ok = mbar_wait(BAR(bqe), nfree, abort_flag, kWaitBudgetNs))) break;
                mbar_expect_tx(BAR(bqf), qbytes);
                for (int a = 0; a < nka; ++a) tma_load_2d(sbase + qbuf_of(c) + a * 8192u, &tmQ, h * dk + 32 * a, y, BAR(bqf));
                if (c >= 2 && !(ok = mbar_wait(BAR(b_kvempty(s)), nfree, abort_flag, kWaitBudgetNs))) break;
                mbar_expect_tx(BAR(b_kvfull(s)), qbytes);
                for (int a = 0; a < nka; ++a)
                    tma_load_2d(sbase + kbuf_of(s) + a * 8192u, &tmK, h * dk + 32 * a, y, BAR(b_kvfull(s)));
                const int bvf = s ? B_VFULL1 : B_VFULL0, bve = s ? B_VEMPTY1 : B_VEMPTY0;
                if (c >= 1 && !(ok = mbar_wait(BAR(bve), (uint32_t)((c - 1) >> 1) & 1u, abort_flag, kWaitBudgetNs))) break;
                mbar_expect_tx(BAR(bvf), kvbytes - qbytes);
                for (int a = 0; a < nva; ++a)
                    tma_load_2d(sbase + vbuf_of(s) + a * 16384u, &tmV, h * dv + 64 * a, y, BAR(bvf));
            }
            for (int c = 0; c < nchunks && ok && !kFull; ++c) {
                const int s = stg(c);
                const int y = row0 + nat(c) * kC;
                if (c >= kNst) ok = mbar_wait(BAR(b_kvempty(s)), ((c / kNst) - 1) & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                mbar_expect_tx(BAR(b_kvfull(s)), kvbytes);
                const uint32_t kdst = sbase + kbuf_of(s), vdst = sbase + vbuf_of(s);
                for (int a = 0; a < nka; ++a) tma_load_2d(kdst + a * 8192u, &tmK, h * dk + 32 * a, y, BAR(b_kvfull(s)));
                for (int a = 0; a < nva; ++a) tma_load_2d(vdst + a * 16384u, &tmV, h * dv + 64 * a, y, BAR(b_kvfull(s)));
                if (!state_only) {
                    if (c >= 1) ok = mbar_wait(BAR(B_QEMPTY), (c - 1) & 1, abort_flag, kWaitBudgetNs);
                    if (!ok) break;
                    mbar_expect_tx(BAR(B_QFULL), qbytes);
                    for (int a = 0; a < nka; ++a)
                        tma_load_2d(sbase + o_q + a * 8192u, &tmQ, h * dk + 32 * a, y, BAR(B_QFULL));
                }
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
            // operand descriptors of the full passes' tiles (the state copy of chunk c sits in the V tile
            // of chunk c - 1)
            const uint64_t dq0 = desc_qk(sbase + o_q), dq1 = desc_qk(sbase + o_q1);
            const uint64_t dk0 = desc_qk(sbase + o_k0), dk1 = desc_qk(sbase + o_k1);
            const uint64_t dkt0 = desc_kt(sbase + o_k0), dkt1 = desc_kt(sbase + o_k1);
            const uint64_t dv0 = desc_v(sbase + o_v0), dv1 = desc_v(sbase + o_v1);
            const uint64_t ds_in_v0 = desc_s(sbase + o_v0, dk), ds_in_v1 = desc_s(sbase + o_v1, dk);
            // image of the state before chunk 0 of this chain (slot start / 128 + seq; chunk c adds c slots)
            // image slot of the state before this segment's first chunk (sequence slot start / 128 + seq,
            // plus the segment's first chunk)
            __nv_bfloat16 *img0 = nullptr;
            if (write_images || save_images) {
                const int ws = blockIdx.x % P.grid_seg;
                const int64_t first_chunk = P.nseg > 1 ? (int64_t)(rev ? P.nseg - 1 - ws : ws) * P.seg_chunks : 0;
                img0 = P.chunk_states + ((rng.start / kC + seq + first_chunk) * H + h) * sz_state;
            }
            bool ok = true;
            for (int c = 0; c < nchunks && ok; ++c) {
                const int s = stg(c);
                const uint32_t kbuf = sbase + kbuf_of(s), vbuf = sbase + vbuf_of(s);
                if (framed) {
                    ok = mbar_wait(BAR(b_kvfull(s)), sph(c), abort_flag, kWaitBudgetNs) &&
                         mbar_wait(BAR(b_kprep(s)), sph(c), abort_flag, kWaitBudgetNs) &&
                         mbar_wait(BAR(B_SREADY), c & 1, abort_flag, kWaitBudgetNs);
                    if (!ok) break;
                    tc_fence_after();
                    mma_group_kv(tmem + kColS, desc_kt(kbuf), desc_v(vbuf), id_kv);
                    mma_commit(BAR(B_SFULL));
                    mma_commit(BAR(b_kvempty(s)));
                    // the image of the state before this chunk: copy it out while the MMA runs
                    bulk_store_s2g(img0 + (int64_t)nat(c) * H * sz_state, sbase + o_s, (uint32_t)(sz_state * 2));
                    bulk_commit();
                    bulk_wait_read0();
                    mbar_arrive(BAR(B_IMGDONE));
                    continue;
                }
                if (blocked) {
                    // pass 1 in frame blocks: a state pass only before the first chunk of each block
                    const int m = c % nblk;
                    const bool block_end = (m == nblk - 1) || (c == nchunks - 1);
                    ok = mbar_wait(BAR(b_kvfull(s)), sph(c), abort_flag, kWaitBudgetNs) &&
                         mbar_wait(BAR(b_kprep(s)), sph(c), abort_flag, kWaitBudgetNs) &&
                         (m != 0 || mbar_wait(BAR(B_SREADY), (c / nblk) & 1, abort_flag, kWaitBudgetNs));
                    if (!ok) break;
                    tc_fence_after();
                    mma_group_kv(tmem + kColS, desc_kt(kbuf), desc_v(vbuf), id_kv);
                    mma_commit(BAR(b_kvempty(s)));
                    if (block_end) mma_commit(BAR(B_SFULL));
                    continue;
                }
                if (state_only) {
                    // pass 1: only the state chain, S += K~^T V per chunk
                    ok = mbar_wait(BAR(b_kvfull(s)), sph(c), abort_flag, kWaitBudgetNs) &&
                         mbar_wait(BAR(b_kprep(s)), sph(c), abort_flag, kWaitBudgetNs) &&
                         mbar_wait(BAR(B_SREADY), c & 1, abort_flag, kWaitBudgetNs);
                    if (!ok) break;
                    tc_fence_after();
                    if (write_images) {
                        // the state in force before chunk nat(c), as the bf16 tile the state pass just
                        // wrote: copy it out, and let it be read before MMA4 (and so before the next state
                        // pass may refill it)
                        bulk_store_s2g(img0 + (int64_t)nat(c) * H * sz_state, sbase + o_s, (uint32_t)(sz_state * 2));
                        bulk_commit();
                        bulk_wait_read0();
                    }
                    mma_group_kv(tmem + kColS, desc_kt(kbuf), desc_v(vbuf), id_kv);
                    mma_commit(BAR(B_SFULL));
                    mma_commit(BAR(b_kvempty(s)));
                    continue;
                }
                // full passes: MMA1(c), MMA3(c), MMA2(c), MMA4(c).  MMA4 last: the state pass of the next
                // chunk waits for it and then writes its copy into V tile c, which MMA2 has read by then.
                const uint64_t dq = (c & 1) ? dq1 : dq0, dkk = s ? dk1 : dk0, dkt = s ? dkt1 : dkt0;
                const uint64_t dvv = s ? dv1 : dv0, dss = (c & 1) ? ds_in_v0 : ds_in_v1;
                const uint32_t sbuf = sbase + scopy_of(c);
                const uint32_t ph = (uint32_t)(c >> 1) & 1u;  // phase of chunk c on its Q tile and K/V stage
                // (factored form: KPREP implies that K has landed)
                ok = mbar_wait(BAR(s ? B_QFULL1 : B_QFULL), ph, abort_flag, kWaitBudgetNs) &&
                     (fact ? mbar_wait(BAR(b_kprep(s)), ph, abort_flag, kWaitBudgetNs)
                           : mbar_wait(BAR(b_kvfull(s)), ph, abort_flag, kWaitBudgetNs));
                if (!ok) break;
                tc_fence_after();
                // MMA1: A = Q K^T, K'' in the factored form (both K-major, 64B swizzle; 2 K-steps per atom)
                mma_group_qk(tmem + kColA, dq, dkk, id_qk, ksteps_dk);
                mma_commit(BAR(B_AFULL));
                ok = mbar_wait(BAR(B_SREADY), c & 1, abort_flag, kWaitBudgetNs);  // copy S_{c-1} ready, O free
                if (!ok) break;
                tc_fence_after();
                if (save_images) {  // the state copy S_{c-1} just written: out to its image slot
                    bulk_store_s2g(img0 + (int64_t)c * H * sz_state, sbuf, (uint32_t)(sz_state * 2));
                    bulk_commit();
                }
                // MMA3: O = Q S_{c-1} (factored) or Q' S_{c-1} (direct); A K-major 64B swizzle,
                // B = S copy, MN-major 128B swizzle
                mma_group_qs(tmem + kColO, dq, dss, id_qs, ksteps_dk);
                mma_commit(BAR(s ? B_QEMPTY1 : B_QEMPTY));    // Q(c+2) may land in this Q tile
                mma_commit(BAR(s ? B_VEMPTY0 : B_VEMPTY1));   // V(c+1) may land over the copy S_{c-1}
                ok = mbar_wait(BAR(s ? B_VFULL1 : B_VFULL0), ph, abort_flag, kWaitBudgetNs) &&
                     mbar_wait(BAR(B_PFULL), c & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
                // MMA2: O += P V (A = P in TMEM, 8 columns per K-step of 16 tokens)
                mma_group_pv(tmem + kColO, tmem + kColA, dvv, id_pv);
                mma_commit(BAR(B_OFULL));
                if (!fact) {
                    ok = mbar_wait(BAR(b_kprep(s)), ph, abort_flag, kWaitBudgetNs);
                    if (!ok) break;
                    tc_fence_after();
                }
                // MMA4: S += K~^T V (A MN-major 64B swizzle over dk, B MN-major 128B swizzle over dv)
                mma_group_kv(tmem + kColS, dkt, dvv, id_kv);
                mma_commit(BAR(B_SFULL));        // after MMA2 as well: V tile c may take the next state copy
                mma_commit(BAR(b_kvempty(s)));   // MMA1 and MMA4 were the readers of this K tile
                if (save_images) {  // V(c+1) may land once the image store has read the copy
                    bulk_wait_read0();
                    mbar_arrive(BAR(s ? B_VEMPTY0 : B_VEMPTY1));
                }
            }
            if (save_images || write_images) bulk_wait_read0();  // no image store may still read shared memory
            if (!ok) {
                record_status(GLA_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ state warpgroup
        const int r = threadIdx.x;                          // TMEM lane = dk row of S = tile row for prep
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        bool ok = true;
        // K rows scaled as soon as K_c lands (no MMA1 reads them first): factored form K''_c rows =
        // lambda^-(j+1) k_j; state-only pass in the direct form K~_c rows = lambda^(L-1-j) k_j.
        // Rows beyond the chunk are zeroed.
        const bool early_k = fact || state_only;
        auto prep_k_early = [&](int c) -> bool {
            if (!mbar_wait(BAR(b_kvfull(stg(c))), sph(c), abort_flag, kWaitBudgetNs)) return false;
            const int Lk = plen(c);
            // forwards: lambda^-(j+1) (factored) or lambda^(L-1-j); backwards in time the weight of row i
            // is lambda^(i+1): lambda^(i+1-L) in the factored form (the state is scaled by lambda^L after)
            const float fw = fact ? utab[r] : tab[Lk - 1 - r];
            const float bw = fact ? tab[min(r + 1, kC)] * utab[Lk - 1] : tab[min(r + 1, kC)];
            const float f = (r < Lk) ? (rev ? bw : fw) : 0.f;
            scale_row_sw64(smem + kbuf_of(stg(c)), nka, r, f);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(b_kprep(stg(c))));
            return true;
        };
        if (framed) {
            // rows walked in the current frame block before the c-th chunk (only the first chunk walked
            // backwards, the sequence's last, can be short; walked forwards the short one comes last)
            auto rows_before = [&](int c) -> int {
                const int m = c % nblk;
                return m * kC - ((rev && c > 0 && c < nblk) ? (kC - plen(0)) : 0);
            };
            // K-role rows of the c-th chunk walked, with their frame factor; rows beyond it zeroed
            auto prep_k_framed = [&](int c) -> bool {
                if (!mbar_wait(BAR(b_kvfull(stg(c))), sph(c), abort_flag, kWaitBudgetNs)) return false;
                const int Lk = plen(c);
                const int e = rows_before(c) + (rev ? Lk - r - 1 : r + 1);
                scale_row_sw64(smem + kbuf_of(stg(c)), nka, r, (r < Lk) ? expf(-ld * (float)e) : 0.f);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(b_kprep(stg(c))));
                return true;
            };
            if (nchunks > 0) ok = prep_k_framed(0);
            int walked = 0;  // rows walked in the current block before the c-th chunk
            for (int c = 0; c <= nchunks && ok; ++c) {
                const bool last = c == nchunks;
                const bool block_start = c > 0 && (c % nblk == 0 || last);  // the previous block just ended
                if (c >= 1) {
                    ok = mbar_wait(BAR(B_SFULL), (c - 1) & 1, abort_flag, kWaitBudgetNs);
                    // the previous image must be out of shared memory before the copy is refilled
                    if (ok && !last) ok = mbar_wait(BAR(B_IMGDONE), (c - 1) & 1, abort_flag, kWaitBudgetNs);
                    if (!ok) break;
                    tc_fence_after();
                }
                // state before the c-th chunk: lambda^walked * frame; at a block start the frame is
                // brought back to the true state (TMEM rewritten) and walked restarts at 0
                const uint64_t g2 = f32x2_splat(expf(ld * (float)walked));
                if (r < dk) {
                    for (int j0 = 0; j0 < dv; j0 += 64) {
                        uint32_t v[2][32];
                        if (c >= 1) {
                            tmem_ld32(tmem + lane_base + kColS + (uint32_t)j0, v[0]);
                            tmem_ld32(tmem + lane_base + kColS + (uint32_t)j0 + 32u, v[1]);
                            tmem_wait_ld();
                            scale32(v[0], g2);
                            scale32(v[1], g2);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                v[0][e] = __float_as_uint(init_state ? __ldg(init_state + (int64_t)r * dv + j0 + e) : 0.f);
                                v[1][e] = __float_as_uint(init_state ? __ldg(init_state + (int64_t)r * dv + j0 + 32 + e) : 0.f);
                            }
                        }
                        if (last) {
                            if (final_state) {
                                float4 *dst = reinterpret_cast<float4 *>(final_state + (int64_t)r * dv + j0);
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    dst[e] = make_float4(__uint_as_float(v[e >> 3][4 * (e & 7)]),
                                                         __uint_as_float(v[e >> 3][4 * (e & 7) + 1]),
                                                         __uint_as_float(v[e >> 3][4 * (e & 7) + 2]),
                                                         __uint_as_float(v[e >> 3][4 * (e & 7) + 3]));
                            }
                            continue;
                        }
                        if (c == 0 || block_start) {
                            tmem_st32(tmem + lane_base + kColS + (uint32_t)j0, v[0]);
                            tmem_st32(tmem + lane_base + kColS + (uint32_t)j0 + 32u, v[1]);
                        }
                        // bf16 image into the MN-major, 128B-swizzled tile: one 64-column atom
                        uint8_t *atom_row = smem + o_s + (uint32_t)(j0 >> 6) * (uint32_t)dk * 128u + (uint32_t)r * 128u;
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8) {
                            const uint32_t *x = &v[q8 >> 2][8 * (q8 & 3)];
                            *reinterpret_cast<uint4 *>(atom_row + (((uint32_t)q8 ^ (uint32_t)(r & 7)) << 4)) =
                                make_uint4(pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                           pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                           pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                           pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
                        }
                    }
                }
                if (last) break;
                if (block_start) walked = 0;
                tmem_wait_st();
                fence_async_shared();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_SREADY));
                walked += plen(c);
                if (c + 1 < nchunks) ok = prep_k_framed(c + 1);
            }
            if (!ok) {
                record_status(GLA_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        } else if (blocked) {
            // K rows of chunk c (m-th of its block): lambda^-(m*128 + j + 1) k_j, rows beyond it zeroed
            // rows walked in the current frame block before the c-th chunk (walked backwards only the
            // first chunk, the sequence's last, can be short; walked forwards the short one comes last)
            auto rows_before = [&](int c) -> int {
                return (c % nblk) * kC - ((rev && c > 0 && c < nblk) ? (kC - plen(0)) : 0);
            };
            auto prep_k_frame = [&](int c) -> bool {
                if (!mbar_wait(BAR(b_kvfull(stg(c))), sph(c), abort_flag, kWaitBudgetNs)) return false;
                const int Lk = plen(c);
                float f;
                if (rev) {  // row i of a chunk walked backwards: lambda^-(rows before it in the block + L - i - 1)
                    f = expf(-ld * (float)(rows_before(c) + Lk - r - 1));
                } else {    // row j walked forwards: lambda^-(128 m + j + 1)
                    f = utab[r] * expf(-ld * (float)((c % nblk) * kC));
                }
                scale_row_sw64(smem + kbuf_of(stg(c)), nka, r, (r < Lk) ? f : 0.f);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(b_kprep(stg(c))));
                return true;
            };
            // the starting state into TMEM
            if (r < dk) {
                for (int j0 = 0; j0 < dv; j0 += 32) {
                    uint32_t v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = __float_as_uint(init_state ? __ldg(init_state + (int64_t)r * dv + j0 + e) : 0.f);
                    tmem_st32(tmem + lane_base + kColS + (uint32_t)j0, v);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_SREADY));
            if (nchunks > 0) ok = prep_k_frame(0);
            for (int c = 0; c < nchunks && ok; ++c) {
                if (c + 1 < nchunks) ok = prep_k_frame(c + 1);
                if (!ok) break;
                const int m = c % nblk;
                if (m != nblk - 1 && c != nchunks - 1) continue;
                // block end: S = lambda^(rows of the block) * (TMEM frame)
                ok = mbar_wait(BAR(B_SFULL), (c / nblk) & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
                const bool last = c == nchunks - 1;
                const uint64_t g2 = f32x2_splat(expf(ld * (float)(rows_before(c) + plen(c))));
                if (r < dk) {
                    for (int j0 = 0; j0 < dv; j0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_base + kColS + (uint32_t)j0, v);
                        tmem_wait_ld();
                        scale32(v, g2);
                        if (last) {
                            if (final_state) {
                                float4 *dst = reinterpret_cast<float4 *>(final_state + (int64_t)r * dv + j0);
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                         __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                            }
                        } else {
                            tmem_st32(tmem + lane_base + kColS + (uint32_t)j0, v);
                        }
                    }
                }
                if (!last) {
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(B_SREADY));
                }
            }
            if (nchunks == 0 && final_state && r < dk) {
                for (int j = 0; j < dv; ++j) final_state[(int64_t)r * dv + j] = init_state ? init_state[(int64_t)r * dv + j] : 0.f;
            }
            if (!ok) {
                record_status(GLA_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        } else {
        if (early_k && nchunks > 0) ok = prep_k_early(0);
        for (int c = 0; c <= nchunks && ok; ++c) {
            if (c >= 1) {
                // (full passes: MMA4(c-1) is issued after MMA2(c-1), so V tile c-1 is free for the copy)
                ok = mbar_wait(BAR(B_SFULL), (c - 1) & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
            }
            const bool last = (c == nchunks);
            // factored: TMEM holds S_{c-2} + K''^T V, S_{c-1} = lambda^L(c-1) * that; copy and TMEM both get it.
            // direct:   TMEM holds S_{c-1}; the copy is S_{c-1}, TMEM gets lambda^L(c) S_{c-1} for MMA4.
            const float g_prev = (fact && c >= 1) ? tab[plen(c - 1)] : 1.f;
            const float g_copy = g_prev;
            const float g_tmem = fact ? g_prev : (last ? 1.f : tab[plen(c)]);
            const uint64_t gc2 = f32x2_splat(g_copy);
            if (r < dk) {
                // two 32-column groups per step: both TMEM loads in flight before the first use
                for (int j0 = 0; j0 < dv; j0 += 64) {
                    uint32_t v[2][32];
                    if (c >= 1) {
                        tmem_ld32(tmem + lane_base + kColS + (uint32_t)j0, v[0]);
                        tmem_ld32(tmem + lane_base + kColS + (uint32_t)j0 + 32u, v[1]);
                        tmem_wait_ld();
                    } else {
                        const float4 *src = reinterpret_cast<const float4 *>(init_state + (int64_t)r * dv + j0);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float4 x = init_state ? __ldg(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                            v[e >> 3][4 * (e & 7)] = __float_as_uint(x.x);
                            v[e >> 3][4 * (e & 7) + 1] = __float_as_uint(x.y);
                            v[e >> 3][4 * (e & 7) + 2] = __float_as_uint(x.z);
                            v[e >> 3][4 * (e & 7) + 3] = __float_as_uint(x.w);
                        }
                    }
                    scale32(v[0], gc2);
                    scale32(v[1], gc2);
                    if (last) {
                        if (final_state) {
                            float4 *dst = reinterpret_cast<float4 *>(final_state + (int64_t)r * dv + j0);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                dst[e] = make_float4(__uint_as_float(v[e >> 3][4 * (e & 7)]),
                                                     __uint_as_float(v[e >> 3][4 * (e & 7) + 1]),
                                                     __uint_as_float(v[e >> 3][4 * (e & 7) + 2]),
                                                     __uint_as_float(v[e >> 3][4 * (e & 7) + 3]));
                        }
                        continue;
                    }
                    // bf16 copy into the MN-major, 128B-swizzled S tile: one 64-column atom
                    uint8_t *atom_row = smem + scopy_of(c) + (uint32_t)(j0 >> 6) * (uint32_t)dk * 128u + (uint32_t)r * 128u;
#pragma unroll
                    for (int q8 = 0; q8 < 8 && (!state_only || write_images); ++q8) {
                        const uint32_t *x = &v[q8 >> 2][8 * (q8 & 3)];
                        *reinterpret_cast<uint4 *>(atom_row + (((uint32_t)q8 ^ (uint32_t)(r & 7)) << 4)) =
                            make_uint4(pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                       pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                       pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                       pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
                    }
                    if (g_tmem != g_copy || c == 0) {
                        const uint64_t gt2 = f32x2_splat(g_tmem / (c == 0 ? 1.f : g_copy));
                        scale32(v[0], gt2);
                        scale32(v[1], gt2);
                    }
                    tmem_st32(tmem + lane_base + kColS + (uint32_t)j0, v[0]);
                    tmem_st32(tmem + lane_base + kColS + (uint32_t)j0 + 32u, v[1]);
                }
            }
            if (last) break;
            tmem_wait_st();
            fence_async_shared();
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && early_k) mbar_arrive(BAR(B_SREADY));  // (direct form: after the Q prep below)

            if (early_k) {
                if (c + 1 < nchunks) ok = prep_k_early(c + 1);
            } else {
                // direct form: decays of the Q and K rows, in place, once MMA1 has read them
                ok = mbar_wait(BAR(B_AFULL), c & 1, abort_flag, kWaitBudgetNs);
                if (!ok) break;
                tc_fence_after();
                const int Lc = chunk_len(c);
                scale_row_sw64(smem + qbuf_of(c), nka, r, tab[min(r + 1, kC)]);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_SREADY));  // the state copy and Q' are ready for MMA3
                scale_row_sw64(smem + ((c & 1) ? o_k1 : o_k0), nka, r, (r < Lc) ? tab[Lc - 1 - r] : 0.f);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_KPREP0 + (c & 1)));
            }
        }
        if (!ok) {
            record_status(GLA_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        }  // not blocked
    } else if (warp < 8) {
        // ------------------------------------------------------------ mask warpgroup
        const int r = threadIdx.x - 128;                    // TMEM lane = token row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        bool ok = true;
        for (int c = 0; c < nchunks && ok && !state_only; ++c) {
            const int Lc = chunk_len(c);
            // ---- mask: P = bf16(A .* D) ----
            ok = mbar_wait(BAR(B_AFULL), c & 1, abort_flag, kWaitBudgetNs);
            if (!ok) break;
            tc_fence_after();
            {
                const bool row_ok = r < Lc;
                // 32-column blocks in increasing j: P block b (16 TMEM columns) only overwrites
                // A columns this thread has already loaded.
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    uint32_t a[32], p[16];
                    tmem_ld32(tmem + lane_base + kColA + (uint32_t)(32 * b), a);
                    tmem_wait_ld();
                    if (fact) {
                        // the decay already sits in K'' and in the epilogue's row factor: causal mask only,
                        // as one 32-bit mask of the block's kept columns (bit t for column 32 b + t)
                        const int d = r - 32 * b;
                        const uint32_t bits = !row_ok ? 0u : d >= 31 ? 0xffffffffu : d < 0 ? 0u : (2u << d) - 1u;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float x0 = ((bits >> (2 * e)) & 1u) ? __uint_as_float(a[2 * e]) : 0.f;
                            const float x1 = ((bits >> (2 * e + 1)) & 1u) ? __uint_as_float(a[2 * e + 1]) : 0.f;
                            p[e] = pack_bf16x2(x0, x1);
                        }
                    } else {
                        // D_rj = lambda^(r-j): walk j downwards from 32b+31, one factor of lambda per step
                        const int dtop = r - (32 * b + 31);
                        float f = tab[max(dtop, 0)];
#pragma unroll
                        for (int e = 15; e >= 0; --e) {
                            const bool on1 = row_ok && (dtop + (30 - 2 * e) >= 0);
                            const float d1 = on1 ? f : 0.f;
                            f = on1 ? f * lam : f;
                            const bool on0 = row_ok && (dtop + (31 - 2 * e) >= 0);
                            const float d0 = on0 ? f : 0.f;
                            f = on0 ? f * lam : f;
                            p[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * d0, __uint_as_float(a[2 * e + 1]) * d1);
                        }
                    }
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                        ::"r"(tmem + lane_base + kColA + (uint32_t)(16 * b)), "r"(p[0]), "r"(p[1]), "r"(p[2]),
                          "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]), "r"(p[8]), "r"(p[9]), "r"(p[10]),
                          "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]), "r"(p[15])
                        : "memory");
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_PFULL));

        }
        if (!ok) {
            record_status(GLA_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------ epilogue warpgroup
        const int q4 = warp & 3;                            // TMEM lane quadrant of this warp
        const int r = 32 * q4 + lane;                       // TMEM lane = token row
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const float grow = fact ? tab[min(r + 1, kC)] : 1.f;  // lambda^(r+1): the factored row factor
        const uint32_t grow2 = pack_bf16x2(grow, grow);           // the same, as a bf16 pair (gated drain)
        const uint64_t grow_f2 = f32x2_splat(grow);                // and as an f32 pair (ungated drain)
        uint8_t *xp = smem + o_xp + (uint32_t)q4 * 4096u;     // this warp's staging tile: 32 rows x 128 B
        bool ok = true;
        // O is free for the first chunk's MMA3 (the releases of O count toward SREADY, one phase later)
        if (!state_only && nchunks > 0 && lane == 0) mbar_arrive(BAR(B_SREADY));
        for (int c = 0; c < nchunks && ok && !state_only && !kGate; ++c) {
            const int Lc = chunk_len(c);
            // ---- output epilogue: O -> bf16 rows in this warp's 4 KB staging tile (one 64-column
            // group of its 32 rows, laid out as a 128B-swizzled TMA box), then a TMA store per group.
            // Only the staging tile's previous store must have read it before it is refilled, so O
            // leaves TMEM at the pace of the TMEM loads, not of the global stores. ----
            ok = mbar_wait(BAR(B_OFULL), c & 1, abort_flag, kWaitBudgetNs);
            if (!ok) break;
            tc_fence_after();
            const bool full = (Lc == kC);
            for (int j0 = 0; j0 < dv; j0 += 64) {
                uint32_t v[2][32];
                tmem_ld32(tmem + lane_base + kColO + (uint32_t)j0, v[0]);
                tmem_ld32(tmem + lane_base + kColO + (uint32_t)j0 + 32u, v[1]);
                tmem_wait_ld();
                scale32(v[0], grow_f2);
                scale32(v[1], grow_f2);
                if (j0 + 64 >= dv) {  // last TMEM read of O for this chunk: MMA3 of the next chunk may start
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(B_SREADY));
                }
                if (lane == 0) bulk_wait_read0();  // the previous store out of the staging tile has read it
                __syncwarp();
                // own row (lane): 64 columns -> 128 B, 16-byte chunk q8 at q8 ^ (lane & 7)
                uint8_t *myrow = xp + (uint32_t)lane * 128u;
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const uint32_t *x = &v[q8 >> 2][8 * (q8 & 3)];
                    *reinterpret_cast<uint4 *>(myrow + (((uint32_t)q8 ^ (uint32_t)(lane & 7)) << 4)) = make_uint4(
                        pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                        pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                        pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                        pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
                }
                if (full) {
                    fence_async_shared();  // the staged rows must be visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmO, h * dv + j0, row0 + c * kC + 32 * q4, sbase + o_xp + (uint32_t)q4 * 4096u);
                        bulk_commit();
                    }
                } else {
                    // partial chunk: the rows from Lc on belong to the next sequence or lie past the
                    // tensor, so the rows below Lc are stored with plain predicated stores, eight lanes
                    // per row
                    __syncwarp();
                    const int ch = lane & 7;
#pragma unroll 4
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + (lane >> 3), row = 32 * q4 + rr;
                        if (row < Lc) {
                            const uint4 x = *reinterpret_cast<const uint4 *>(
                                xp + (uint32_t)rr * 128u + (((uint32_t)ch ^ (uint32_t)(rr & 7)) << 4));
                            *reinterpret_cast<uint4 *>(P.out + ((row0 + (int64_t)c * kC + row) * H + h) * dv + j0 +
                                                       8 * ch) = x;
                        }
                    }
                    __syncwarp();
                }
            }
        }
        // ---- gated instance: out = O * f(g).  The gate rows of a 64-column group (the warp's 32 rows x
        // 128 bytes) come in with one TMA box into one of two 4 KB buffers, the gate buffer and the staging
        // tile, alternating by group and laid out as the staging tile (the box of the output store); each
        // lane turns its own row of gate values into its row of gated output in place, and the group's TMA
        // store goes out of that buffer.  The first two groups' gates are loaded before O is ready, each
        // later one as soon as the store two groups back has read its buffer; the next chunk's gate lines
        // are prefetched into L2.  Each buffer has its barrier (count 1, the box's bytes). ----
        auto gbar = [&](int b) -> uint32_t { return BAR(B_COUNT + 2 * q4 + b); };
        // gate loads per buffer, issued and waited for (scalars: a runtime index would put them in local memory)
        uint32_t gissued0 = 0u, gissued1 = 0u, gused0 = 0u, gused1 = 0u;
        auto wait_gate = [&](int b) -> bool {
            const uint32_t n = b ? gused1 : gused0;
            const bool landed = mbar_wait(gbar(b), n & 1u, abort_flag, kWaitBudgetNs);
            if (b) ++gused1; else ++gused0;
            return landed;
        };
        for (int c = 0; c < nchunks && ok && kGate; ++c) {
            const int Lc = chunk_len(c);
            const int ng = dv / 64, gk = P.gate_kind;
            auto buf_of = [&](int j) -> uint32_t { return ((j & 1) ? o_xp : o_gb) + (uint32_t)q4 * 4096u; };
            // the gate rows of group j (this warp's 32 rows x 64 columns) with one TMA box, laid out like the
            // output staging; rows past the tensor read as zeros, rows of the next sequence are not stored
            auto load_gate = [&](int j) {
                if (lane == 0) {
                    const uint32_t bar = gbar(j & 1);
                    mbar_expect_tx(bar, 4096u);
                    tma_load_2d(sbase + buf_of(j), &tmG, h * dv + 64 * j, row0 + c * kC + 32 * q4, bar);
                }
                if (j & 1) ++gissued1; else ++gissued0;
            };
            if (c + 1 < nchunks && r < chunk_len(c + 1)) {
                const __nv_bfloat16 *gn = P.gate + ((row0 + (int64_t)(c + 1) * kC + r) * H + h) * dv;
                for (int j0 = 0; j0 < dv; j0 += 64)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(gn + j0)));
            }
            if (lane == 0) bulk_wait_read0();  // both buffers: the previous chunk's stores have read them
            __syncwarp();
            load_gate(0);
            if (ng > 1) load_gate(1);
            ok = mbar_wait(BAR(B_OFULL), c & 1, abort_flag, kWaitBudgetNs);
            if (!ok) break;
            tc_fence_after();
            const bool full = (Lc == kC);
            for (int j = 0; j < ng; ++j) {
                const int j0 = 64 * j;
                uint8_t *myrow = smem + buf_of(j) + (uint32_t)lane * 128u;
                // two 32-column halves (32 registers of O at a time: the gate arithmetic needs the rest)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kColO + (uint32_t)(j0 + 32 * hf), v);
                    if (hf == 0) {
                        // gate j has landed
                        ok = wait_gate(j & 1) && ok;
                        // the gate of group j + 1 goes where group j - 1 was staged, once that store has read it
                        if (j >= 1 && j + 1 < ng) {
                            if (lane == 0) bulk_wait_read0();
                            __syncwarp();
                            load_gate(j + 1);
                        }
                    }
                    tmem_wait_ld();
                    if (j + 1 == ng && hf == 1) {  // last TMEM read of O for this chunk: MMA3 of the next may start
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(BAR(B_SREADY));
                    }
                    // own row (lane): 32 gate values -> 32 gated outputs in place, 16-byte chunk q8 at q8 ^ (lane & 7)
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const int q8 = 4 * hf + qq;
                        uint4 *cell = reinterpret_cast<uint4 *>(myrow + (((uint32_t)q8 ^ (uint32_t)(lane & 7)) << 4));
                        const uint4 gq = *cell;
                        const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
                        const uint32_t *x = &v[8 * qq];
                        uint32_t o2[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // in bf16 pairs: the gate factor times the row factor, times O rounded to bf16
                            uint32_t fg;
                            asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(fg) : "r"(gate_factor_bf16x2(gw[e], gk)), "r"(grow2));
                            asm("mul.rn.bf16x2 %0, %1, %2;"
                                : "=r"(o2[e])
                                : "r"(pack_bf16x2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1]))), "r"(fg));
                        }
                        *cell = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                    }
                }
                if (full) {
                    fence_async_shared();  // the staged rows must be visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmO, h * dv + j0, row0 + c * kC + 32 * q4, sbase + buf_of(j));
                        bulk_commit();
                    }
                } else {
                    // partial chunk: plain predicated stores of the rows below Lc (as in the plain epilogue)
                    __syncwarp();
                    const int ch = lane & 7;
                    const uint8_t *tile = smem + buf_of(j);
#pragma unroll 4
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + (lane >> 3), row = 32 * q4 + rr;
                        if (row < Lc) {
                            const uint4 x = *reinterpret_cast<const uint4 *>(
                                tile + (uint32_t)rr * 128u + (((uint32_t)ch ^ (uint32_t)(rr & 7)) << 4));
                            *reinterpret_cast<uint4 *>(P.out + ((row0 + (int64_t)c * kC + row) * H + h) * dv + j0 +
                                                       8 * ch) = x;
                        }
                    }
                    __syncwarp();
                }
            }
        }
        if (lane == 0) bulk_wait_read0();  // no store may still read shared memory at exit
        // no gate load may still be writing shared memory at exit (after a wait that gave up): bounded waits
        // that do not end on the abort flag
        if (kGate) {
            for (; gused0 < gissued0; ++gused0) mbar_wait(gbar(0), gused0 & 1u, nullptr, kWaitBudgetNs);
            for (; gused1 < gissued1; ++gused1) mbar_wait(gbar(1), gused1 & 1u, nullptr, kWaitBudgetNs);
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
            if (lane == 0) mma_commit(BAR(B_FINAL));
            __syncwarp();
            mbar_wait(BAR(B_FINAL), 0, nullptr, kWaitBudgetNs);
        }
        tmem_dealloc(tmem, kTmemCols);
    }
#undef BAR
}

// Segment start states from the segments' zero-start end states (between pass 1 and pass 2):
//   S_in(0) = h0,  S_in(s+1) = lambda^len(s) S_in(s) + E(s),
// where every segment but the last has the same length.  One thread per 4 state elements.
__global__ void __launch_bounds__(256)
gla_seg_scan_kernel(const float *__restrict__ log_decay, const float *__restrict__ h0,
                    const float *__restrict__ seg_end, float *__restrict__ seg_h0, int H, int dk, int dv,
                    int nseg, int seg_tokens, int first_tokens) {
    const int chain = blockIdx.y, h = chain % H;
    const int64_t sz = (int64_t)dk * dv;
    const int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (e >= sz) return;
    float4 S = h0 ? __ldg(reinterpret_cast<const float4 *>(h0 + chain * sz + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float ld = __ldg(log_decay + h);
    for (int s = 0; s + 1 < nseg; ++s) {
        // walk segment s has seg_tokens rows, except the first walked backwards (first_tokens)
        const float g = expf(ld * (float)(s == 0 ? first_tokens : seg_tokens));
        const int64_t off = ((int64_t)chain * (nseg - 1) + s) * sz + e;
        const float4 E = __ldg(reinterpret_cast<const float4 *>(seg_end + off));
        S.x = fmaf(g, S.x, E.x);
        S.y = fmaf(g, S.y, E.y);
        S.z = fmaf(g, S.z, E.z);
        S.w = fmaf(g, S.w, E.w);
        *reinterpret_cast<float4 *>(seg_h0 + off) = S;
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

}  // namespace

// 2-D bf16 tensor map over [rows, cols] (row stride cols * 2 bytes) with a box of box_rows x box_cols.
bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              CUtensorMapSwizzle sw, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map of any element type over [rows, cols] (row stride cols * elem_bytes), box box_rows x box_cols.
bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base, uint64_t cols,
                 uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * elem_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              CUtensorMapSwizzle sw) {
    return gla::make_map(m, base, cols, rows, box_cols, sw, kC);
}
}  // namespace

bool tc_chunk_supported(int dk, int dv, int chunk) {
    if (!(chunk == kC && dk % 32 == 0 && dk >= 32 && dk <= 128 && dv % 64 == 0 && dv >= 64 && dv <= 192))
        return false;
    const uint32_t cap = (uint32_t)device_info().max_smem_optin;
    return smem_plan(dk, dv).total + 1024 <= cap && smem_plan_full(dk, dv).total + 1024 <= cap;
}

// The gated full pass also needs its 16 KB of gate rows.
bool tc_gate_supported(int dk, int dv) {
    return tc_chunk_supported(dk, dv, kC) &&
           smem_plan_full(dk, dv, true).total + 1024 <= (uint32_t)device_info().max_smem_optin;
}

namespace {

// Segments per chain for a dense batch: as many as fill one wave of CTAs (one per SM), each at
// least kMinSegChunks chunks long; 1 means the whole-chain kernel.
constexpr int kMinSegChunks = 4;

int plan_segments(int nseq, int H, int Tlen, const int32_t *cu, int *seg_chunks) {
    const int nck = (Tlen + kC - 1) / kC;
    *seg_chunks = nck;
    if (cu != nullptr) return 1;
    const long long chains = (long long)nseq * H;
    const int sms = device_info().sm_count;
    if (chains <= 0 || chains * 2 > sms) return 1;
    int nseg = (int)(sms / chains);
    nseg = nseg < nck / kMinSegChunks ? nseg : nck / kMinSegChunks;
    if (nseg < 2) return 1;
    *seg_chunks = (nck + nseg - 1) / nseg;
    return (nck + *seg_chunks - 1) / *seg_chunks;
}

// Bytes of segment-state scratch the segmented schedule takes: the end states from zero and the start
// states, each [chains, nseg - 1, dk, dv] f32.  plan_segments keeps chains * nseg <= SMs, so this is at
// most 2 * (SMs - chains) * dk * dv * 4 < 2 * SMs * dk * dv * 4.
constexpr long long seg_scratch_bytes(long long chains, int nseg, int dk, int dv) {
    return nseg > 1 ? 2LL * chains * (nseg - 1) * dk * dv * 4 : 0;
}

// The largest state (dk * dv) among the head sizes the tensor-core forward takes: dk a multiple of 32 up to
// 128, dv a multiple of 64 up to 192, both shared-memory plans within the 227 KB a CTA may opt in to.
constexpr long long max_tc_state_elems() {
    long long best = 0;
    for (int dk = 32; dk <= 128; dk += 32)
        for (int dv = 64; dv <= 192; dv += 64)
            if (smem_plan(dk, dv).total + 1024 <= 232448u && smem_plan_full(dk, dv).total + 1024 <= 232448u &&
                (long long)dk * dv > best)
                best = (long long)dk * dv;
    return best;
}
// The no-alloc forward's fixed array holds the segment states of every problem the tensor-core kernel takes
// on a GB300 (152 SMs, at least one chain): GLA_ERR_SCRATCH_LIMIT is never returned there.
static_assert(max_tc_state_elems() == 96 * 192, "the largest tensor-core state is 96 x 192");
static_assert(seg_scratch_bytes(1, 152, 96, 192) <= (long long)GLA_NOALLOC_SCRATCH_BYTES,
              "the no-alloc scratch array must hold the segment states of one chain cut over 152 SMs");

// A third K/V stage takes the Q buffer (same size as a K tile) and the state copy plus the output
// staging space for its V tile.
bool three_stages_fit(int dk, int dv) {
    const Smem p = smem_plan(dk, dv);
    return (uint32_t)(dv / 64) * 16384u <= p.tab - p.s;
}

template <bool kRev, int kNst, bool kFull, bool kGate = false>
int launch_one(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
               const CUtensorMap &mg, const Params &p, long long ctas, cudaStream_t st) {
    const size_t bytes = (kFull ? smem_plan_full(p.dk, p.dv, kGate) : smem_plan(p.dk, p.dv)).total + 1024;  // + alignment slack
    if (cudaFuncSetAttribute(gla_tc_chunk_kernel<kRev, kNst, kFull, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bytes) != cudaSuccess)
        return GLA_ERR_LAUNCH;
    gla_tc_chunk_kernel<kRev, kNst, kFull, kGate><<<(unsigned)ctas, kThreads, bytes, st>>>(mq, mk, mv, mo, mg, p);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}

// mg: the output gate's map (gated passes; any valid map otherwise)
int launch_tc(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
              const CUtensorMap &mg, const Params &p, long long ctas, cudaStream_t st) {
    if (ctas <= 0) return GLA_OK;
    if (ctas > 0x7fffffffLL) return GLA_ERR_UNSUPPORTED;
    if (p.mode == kWhole || p.mode == kSegmented)
        return p.gate ? launch_one<false, 2, true, true>(mq, mk, mv, mo, mg, p, ctas, st)
                      : launch_one<false, 2, true, false>(mq, mk, mv, mo, mg, p, ctas, st);
    const bool three = p.mode == kStateOnly && three_stages_fit(p.dk, p.dv);
    if (p.reverse && three) return launch_one<true, 3, false>(mq, mk, mv, mo, mg, p, ctas, st);
    if (p.reverse) return launch_one<true, 2, false>(mq, mk, mv, mo, mg, p, ctas, st);
    if (three) return launch_one<false, 3, false>(mq, mk, mv, mo, mg, p, ctas, st);
    return launch_one<false, 2, false>(mq, mk, mv, mo, mg, p, ctas, st);
}

}  // namespace

// The forward on the tensor cores; with `images` non-null the full passes also leave the bf16 state in
// force before every chunk there ([slots, H, dk, dv], chunk c of sequence s at slot start_s / 128 + s + c).
static int chunk_fwd_impl(const void *q, const void *k, const void *v, const float *ld, const float *h0, void *out,
                   float *hT, void *images, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu,
                   cudaStream_t st, const void *gate = nullptr, int gate_kind = 0) {
    if (!tc_chunk_supported(dk, dv, kC)) return GLA_ERR_UNSUPPORTED;
    const uint64_t rows = cu ? (uint64_t)Tlen : (uint64_t)nseq * (uint64_t)Tlen;
    if (rows >= (1ull << 31)) return GLA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv, mo, mg;
    if (!make_map(&mq, q, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mk, k, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mv, v, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mo, out, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32))
        return GLA_ERR_LAUNCH;
    // the output gate, [rows, H, dv] like out: the same boxes, read by the gated drain
    if (gate == nullptr)
        mg = mo;
    else if (!make_map(&mg, gate, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32))
        return GLA_ERR_LAUNCH;
    Params p{};
    p.log_decay = ld;
    p.h0 = h0;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.hT = hT;
    p.cu = cu;
    p.T = Tlen;
    p.H = H;
    p.dk = dk;
    p.dv = dv;
    p.mode = kWhole;
    p.nseg = 1;
    p.seg_chunks = 0;
    p.grid_seg = 1;
    p.seg_h0 = nullptr;
    p.seg_end = nullptr;
    p.nseq = nseq;
    p.chunk_states = reinterpret_cast<__nv_bfloat16 *>(images);
    p.gate = reinterpret_cast<const __nv_bfloat16 *>(gate);
    p.gate_kind = gate_kind;
    const long long chains = (long long)nseq * H;
    int seg_chunks = 0;
    const int nseg = plan_segments(nseq, H, Tlen, cu, &seg_chunks);
    p.lpt = (cu != nullptr && nseg == 1 && nseq > 1 && nseq <= kLptMaxSeq) ? 1 : 0;
    if (nseg == 1) return launch_tc(mq, mk, mv, mo, mg, p, chains, st);

    // segmented schedule: stream-ordered scratch for the segment end / start states
    const size_t per = (size_t)chains * (size_t)(nseg - 1) * (size_t)dk * (size_t)dv;
    float *scratch = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&scratch), 2 * per * sizeof(float), st) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_NOMEM;
    }
    p.nseg = nseg;
    p.seg_chunks = seg_chunks;
    p.seg_end = scratch;
    p.seg_h0 = scratch + per;
    p.mode = kStateOnly;
    p.grid_seg = nseg - 1;
    p.chunk_states = nullptr;  // the end states from zero are not states of the sequence
    int rc = launch_tc(mq, mk, mv, mo, mg, p, chains * (nseg - 1), st);
    if (rc == GLA_OK) {
        dim3 grid((unsigned)((dk * dv / 4 + 255) / 256), (unsigned)chains);
        gla_seg_scan_kernel<<<grid, 256, 0, st>>>(ld, h0, p.seg_end, scratch + per, H, dk, dv, nseg,
                                                  seg_chunks * kC, seg_chunks * kC);
        count_launches(1);
        rc = cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
    }
    if (rc == GLA_OK) {
        p.mode = kSegmented;
        p.grid_seg = nseg;
        p.chunk_states = reinterpret_cast<__nv_bfloat16 *>(images);
        rc = launch_tc(mq, mk, mv, mo, mg, p, chains * nseg, st);
    }
    cudaFreeAsync(scratch, st);
    return rc;
}

int tc_chunk_fwd_bf16(const void *q, const void *k, const void *v, const float *ld, const float *h0, void *out,
                      float *hT, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu, cudaStream_t st) {
    return chunk_fwd_impl(q, k, v, ld, h0, out, hT, nullptr, nseq, Tlen, H, dk, dv, cu, st);
}

// The forward with the output gate applied to every output row (gate: [rows, H, dv] like out).
int tc_chunk_fwd_gated_bf16(const void *q, const void *k, const void *v, const void *g, int gate_kind, const float *ld,
                            const float *h0, void *out, float *hT, int nseq, int Tlen, int H, int dk, int dv,
                            const int32_t *cu, cudaStream_t st) {
    return chunk_fwd_impl(q, k, v, ld, h0, out, hT, nullptr, nseq, Tlen, H, dk, dv, cu, st, g, gate_kind);
}

int tc_chunk_fwd_bf16_save(const void *q, const void *k, const void *v, const float *ld, const float *h0, void *out,
                           float *hT, void *images, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu,
                           cudaStream_t st) {
    return chunk_fwd_impl(q, k, v, ld, h0, out, hT, images, nseq, Tlen, H, dk, dv, cu, st);
}

// ---- state passes of the backward ------------------------------------------------------
// One state-only walk over every (sequence, head) chain with the tiles of `ka` ([rows, H, dk], in the
// role of k) and `va` ([rows, H, dv], in the role of v): forwards from `init` (or zeros), or backwards
// in time (reverse != 0).  The bf16 state in force before every chunk goes to `images`
// ([slots, H, dk, dv], chunk c of sequence s at slot start_s / 128 + s + c); the final state to
// `final_` if given.  Forwards with (k, v) this yields the S_{c-1}; backwards with (q, dout) from dhT
// the gradient states G_c and dh0.
int tc_state_pass_bf16(const void *ka, const void *va, const float *ld, const float *init, float *final_,
                       void *images, int reverse, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu,
                       cudaStream_t st) {
    if (!tc_chunk_supported(dk, dv, kC)) return GLA_ERR_UNSUPPORTED;
    const uint64_t rows = cu ? (uint64_t)Tlen : (uint64_t)nseq * (uint64_t)Tlen;
    if (rows >= (1ull << 31)) return GLA_ERR_UNSUPPORTED;
    CUtensorMap mk, mv;
    if (!make_map(&mk, ka, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mv, va, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return GLA_ERR_LAUNCH;
    Params p{};
    p.log_decay = ld;
    p.h0 = init;
    p.hT = final_;
    p.cu = cu;
    p.T = Tlen;
    p.H = H;
    p.dk = dk;
    p.dv = dv;
    p.mode = kStates;
    p.nseg = 1;
    p.grid_seg = 1;
    p.reverse = reverse ? 1 : 0;
    p.chunk_states = reinterpret_cast<__nv_bfloat16 *>(images);
    p.nseq = nseq;
    const long long chains = (long long)nseq * H;
    int seg_chunks = 0;
    const int nseg = plan_segments(nseq, H, Tlen, cu, &seg_chunks);
    p.lpt = (cu != nullptr && nseg == 1 && nseq > 1 && nseq <= kLptMaxSeq) ? 1 : 0;
    // the q and out maps are not read in a state-only pass
    if (nseg == 1) return launch_tc(mk, mk, mv, mv, mv, p, chains, st);

    // few long chains: as the forward's segmented schedule, in walk order (backwards in time the first
    // walked segment is the sequence's last, which may be short): end states of walk segments
    // 0..nseg-2 from zero, a scan for the start states, then every segment from its start state
    const size_t per = (size_t)chains * (size_t)(nseg - 1) * (size_t)dk * (size_t)dv;
    float *scratch = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&scratch), 2 * per * sizeof(float), st) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_NOMEM;
    }
    p.nseg = nseg;
    p.seg_chunks = seg_chunks;
    p.seg_end = scratch;
    p.seg_h0 = scratch + per;
    p.mode = kStateOnly;
    p.grid_seg = nseg - 1;
    int rc = launch_tc(mk, mk, mv, mv, mv, p, chains * (nseg - 1), st);
    if (rc == GLA_OK) {
        const int seg_tokens = seg_chunks * kC;
        const int first_tokens = reverse ? Tlen - (nseg - 1) * seg_tokens : seg_tokens;
        dim3 grid((unsigned)((dk * dv / 4 + 255) / 256), (unsigned)chains);
        gla_seg_scan_kernel<<<grid, 256, 0, st>>>(ld, init, p.seg_end, scratch + per, H, dk, dv, nseg, seg_tokens,
                                                  first_tokens);
        count_launches(1);
        rc = cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
    }
    if (rc == GLA_OK) {
        p.mode = kStates;
        p.grid_seg = nseg;
        rc = launch_tc(mk, mk, mv, mv, mv, p, chains * nseg, st);
    }
    cudaFreeAsync(scratch, st);
    return rc;
}

// ---- no-alloc variant ------------------------------------------------------------
// Segment-state scratch that is part of the module image: callers of gla_chunk_fwd_noalloc
// cannot let the library allocate, so the segmented schedule uses this array instead of
// cudaMallocAsync.  Host code must not pass the symbol itself to a kernel (in host code it
// is a host-side stand-in); the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[GLA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
std::atomic<float *> g_scratch_ptr[kMaxDev];  // set once a lookup on that device has succeeded

// Device address of the scratch array on the current device.  A successful lookup is kept for the
// process; a failed one is not: its CUDA error is cleared (so that no later, unrelated call reports it)
// and the next call tries again.  With lazy module loading the lookup is what loads this file's kernels
// and the array onto the device when no other entry point has, so it can fail for want of memory:
// that is GLA_ERR_NOMEM, any other failure GLA_ERR_LAUNCH.
float *noalloc_scratch(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        *err = GLA_ERR_LAUNCH;
        return nullptr;
    }
    float *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            void *addr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
            if (e != cudaSuccess || addr == nullptr) {
                cudaGetLastError();
                *err = (e == cudaErrorMemoryAllocation) ? GLA_ERR_NOMEM : GLA_ERR_LAUNCH;
                return nullptr;
            }
            p = static_cast<float *>(addr);
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *err = GLA_OK;
    return p;
}
}  // namespace

// Same schedule as tc_chunk_fwd_bf16; only the segment-state scratch comes from the static array.
int tc_chunk_fwd_bf16_noalloc(const void *q, const void *k, const void *v, const float *ld, const float *h0,
                              void *out, float *hT, int nseq, int Tlen, int H, int dk, int dv, const int32_t *cu,
                              cudaStream_t st) {
    if (!tc_chunk_supported(dk, dv, kC)) return GLA_ERR_UNSUPPORTED;
    const long long chains = (long long)nseq * H;
    int seg_chunks = 0;
    const int nseg = plan_segments(nseq, H, Tlen, cu, &seg_chunks);
    if (nseg == 1) return tc_chunk_fwd_bf16(q, k, v, ld, h0, out, hT, nseq, Tlen, H, dk, dv, cu, st);  // no scratch
    const size_t per = (size_t)chains * (size_t)(nseg - 1) * (size_t)dk * (size_t)dv;
    if (seg_scratch_bytes(chains, nseg, dk, dv) > (long long)GLA_NOALLOC_SCRATCH_BYTES) return GLA_ERR_SCRATCH_LIMIT;
    int err = GLA_OK;
    float *scratch = noalloc_scratch(&err);
    if (!scratch) return err;

    const uint64_t rows = (uint64_t)nseq * (uint64_t)Tlen;
    if (rows >= (1ull << 31)) return GLA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, q, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mk, k, (uint64_t)H * dk, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&mv, v, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mo, out, (uint64_t)H * dv, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32))
        return GLA_ERR_LAUNCH;
    Params p{};
    p.log_decay = ld;
    p.h0 = h0;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.hT = hT;
    p.cu = cu;
    p.T = Tlen;
    p.H = H;
    p.dk = dk;
    p.dv = dv;
    p.nseg = nseg;
    p.seg_chunks = seg_chunks;
    p.seg_end = scratch;        // written in full by pass 1 before the scan reads it
    p.seg_h0 = scratch + per;   // written in full by the scan before pass 2 reads it
    p.mode = kStateOnly;
    p.grid_seg = nseg - 1;
    int rc = launch_tc(mq, mk, mv, mo, mo, p, chains * (nseg - 1), st);
    if (rc != GLA_OK) return rc;
    dim3 grid((unsigned)((dk * dv / 4 + 255) / 256), (unsigned)chains);
    gla_seg_scan_kernel<<<grid, 256, 0, st>>>(ld, h0, p.seg_end, scratch + per, H, dk, dv, nseg, seg_chunks * kC,
                                              seg_chunks * kC);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return GLA_ERR_LAUNCH;
    p.mode = kSegmented;
    p.grid_seg = nseg;
    return launch_tc(mq, mk, mv, mo, mo, p, chains * nseg, st);
}

}  // namespace gla
