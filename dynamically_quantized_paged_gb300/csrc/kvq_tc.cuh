// kvq_tc.cuh -- split-K fused-dequantization paged GQA decode attention (K2)
// on the fifth-generation tensor cores (tcgen05), with the split merge fused
// into its end.
//
// What it computes ("What is KV Cache Optimization? ...", section "Technical
// Architecture", stage "Fused Dequantization Attention Kernel"; "Dynamic KV
// Cache Quantization for Fast LLM Inference", section "Recap of KV Caching"):
// for sequence b and query head g (KV head h = g / G), softmax over every
// cached token t < seq_len of <q, K_t> / sqrt(d), applied to V_t, where K_t and
// V_t are dequantized from their codes inside the kernel and the pages of the
// sequence are found through its block table.
//
// Why tensor cores.  The G query heads that share a KV head read the same
// codes: per 128-token tile the scores are a [128 x d] x [d x G] product and
// the values a [d x 128] x [128 x G] product.  On the CUDA cores that is G
// multiply-adds per code byte for each of the two (2G at 16-bit query
// precision), which at G = 8 takes longer than streaming the bytes from HBM.
// Here the codes are widened exactly to fp16 (every INT8, E4M3 and INT4 code
// is an fp16 value) and both products run as tcgen05.mma kind::f16 with fp32
// accumulation; the CUDA cores only widen codes, run the online softmax and
// fold the per-token scales in.
//
// One CTA per SM (persistent grid), 12 warps:
//  * warps 8-10, the producers: stream each tile's pages with 16-byte
//    cp.async into a ring of R raw stages (K codes, V codes, scales, INT4
//    zero-points, the piece's query rows), the tile's 16-token units dealt
//    round-robin over the three warps; completion is tracked by the stage's
//    mbarrier (cp.async.mbarrier.arrive), so no producer waits for its
//    copies, and the page ids of the next tile are loaded while the copies
//    of this one are issued;
//  * warps 0-3, the token group (thread = token of the tile): widens its
//    token's K codes into tensor memory (the A operand of the scores, lane =
//    token), builds the query operand at the start of each piece, and after
//    the scores MMA runs the online softmax for its token: per-token scales,
//    tile maxima, exponentials, and the fp16 weights W (the B operand of the
//    values MMA);
//  * warps 4-7, the channel group: widens each token's V codes into shared
//    memory (the A operand of the values MMA, stored channel-contiguous per
//    token: "MN-major"), then, thread = channel, folds each tile's values
//    product into its running fp32 output (rescaled by the softmax's alpha);
//  * warp 11, lane 0, the MMA issuer: scores of tile i, then values of tile
//    i - 1, each completed into an mbarrier by tcgen05.commit.
// Every operand buffer is double-buffered by tile parity, so the token group
// widens tile i + 1 while the scores of tile i run, and the channel group
// widens V of tile i + 1 while the values of tile i run.  All waits are
// bounded (a timeout flags KVQ_ERR_DEVICE_TIMEOUT and the CTA stops working,
// drains its tensor-core work, frees its tensor memory and exits).
//
// Numerics.  INT8 scores: the query is 16-bit fixed point per head (q ~ sq
// (256 hi + lo), hi signed, lo unsigned bytes), the MMA forms the hi and lo
// dot products as exact integers in fp32 (|sum| < 2^24), and the score is
// sq * k_scale * (256 hi + lo).  FP8 scores: fp16 query (exact from bf16 in
// range) against exactly widened E4M3 codes.  INT4 scores: the hi/lo
// fixed-point query split per 32-channel group (block-diagonal operand, so
// each group's dot is exact), with the group's scale and zero-point applied
// to its dot.  Values: W = p * v_scale / max(v_scale over the tile) in fp16
// (at most 1; relative rounding 2^-12), times the exactly widened codes; the
// tile's factor max(v_scale) and the running softmax rescale are applied in
// fp32 (INT4: per-group scales enter W, the zero-point term sum_t p v_zero
// is kept per thread in fp32).
#pragma once

#include <atomic>

#include "kvq_decode.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace tc {

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t a, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    return done != 0;
}
// Potentially blocking test: the thread may be suspended until the phase
// completes or about SUSPEND_NS have passed (rather than for a system-defined
// time), which bounds the polling of a long wait.
constexpr uint32_t SUSPEND_NS = 1000000;
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity), "r"(SUSPEND_NS)
        : "memory");
    return done != 0;
}
// Waits for the completion of the phase with the given parity, for at most
// about two seconds; a timeout flags the error word and returns false.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
static __device__ __noinline__ bool mbar_wait_slow(uint32_t a, uint32_t parity, unsigned* err) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try(a, parity)) {
        if (globaltimer() - t0 > WAIT_LIMIT_NS) {
            flag_error(err, ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, unsigned* err) {
    if (mbar_test(a, parity)) return true;
    return mbar_wait_slow(a, parity, err);
}
// The mbarrier receives one arrival once every cp.async this thread issued
// before has completed (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t a) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: start address, leading
// (K-direction) and stride (M/N-direction) byte offsets between 8 x 16-byte
// core matrices; bit 46 is the descriptor version.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}
// Instruction descriptor, kind::f16: fp16 A and B, fp32 accumulator, M x N,
// A / B K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_smem_a(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Named barrier among the token group's 128 threads; returns whether any of
// them passed `flag`.
__device__ __forceinline__ bool tg_barrier_any(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, 1, 128, p;\n\tselp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)flag)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void tg_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// fp16 pairs of codes.  INT8: 0x64XX is 1024 + XX, so (code + 128) in the low
// byte then minus 1152 gives the code exactly.
__device__ __forceinline__ void s8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&x);
    hi = *reinterpret_cast<const uint32_t*>(&y);
}
// INT4: eight nibbles (channels 8i..8i+7, low nibble first) -> four fp16
// pairs (n0, n4), (n1, n5), (n2, n6), (n3, n7), each 1024 + nibble.
__device__ __forceinline__ uint32_t nib_pair(uint32_t w) {
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(d) : "r"(w));
    return d;
}
// The channel held at K-position p (0..7) of an 8-channel block of INT4 codes.
__host__ __device__ constexpr int int4_perm8(int p) { return (p & 1) ? (p >> 1) + 4 : (p >> 1); }

// XOR-swizzled position of 16-byte chunk L of a raw code tile (row-major
// chunks): within each 128-byte line the slot is XORed with the line index,
// so that a warp reading one chunk of 8 consecutive rows hits 8 banks groups.
__device__ __forceinline__ int swz(int L) { return (L & ~7) | ((L ^ (L >> 3)) & 7); }

// float -> int key whose signed order is the float order (no NaNs).
__device__ __forceinline__ int fkey(float f) {
    const int b = __float_as_int(f);
    return b ^ ((b >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float fkey_inv(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF)); }

// ---------------------------------------------------------------- configuration
template <int SCHEME, int D, int G>
struct Cfg {
    // the per-channel K scheme is INT8 whose widened K columns are also
    // multiplied by the page's channel factors (KCH)
    static constexpr bool INT8 = SCHEME == KVQ_INT8_SYM_TOKEN || SCHEME == KVQ_INT8_KCHAN;
    static constexpr bool KCH = SCHEME == KVQ_INT8_KCHAN;
    static constexpr bool FP8 = SCHEME == KVQ_FP8E4M3_TOKEN;
    // both INT4 schemes share the 4-bit layout and the group arithmetic; the
    // symmetric one has fp32 scales, no stored zero-point (zero = -8 scale
    // once its two's-complement codes are read as offset binary, code ^ 8)
    static constexpr bool INT4 = SCHEME == KVQ_INT4_ASYM_G32 || SCHEME == KVQ_INT4_SYM_G32;
    static constexpr bool SYM4 = SCHEME == KVQ_INT4_SYM_G32;
    static constexpr uint32_t NIBX = SYM4 ? 0x88888888u : 0u;  // XOR taking codes to offset binary
    static constexpr int T = 128;                  // tokens per tile
    static constexpr int TU = T / UNIT;            // 16-token units per tile
    static constexpr int CB = INT4 ? D / 2 : D;    // code bytes per token row
    static constexpr int NCH = CB / 16;            // 16-byte chunks per token row
    static constexpr int NGR = D / 32;             // INT4 groups per row
    static constexpr int MB = INT4 ? NGR * (SYM4 ? 4 : 2) : 4;  // bytes per token in one scale (or zero) array
    // scores MMA columns: INT8 hi | lo per head; FP8 one per head; INT4 hi | lo per (group, head)
    static constexpr int NS_USED = INT8 ? 2 * G : (INT4 ? 2 * NGR * G : G);
    static constexpr int NS = NS_USED <= 16 ? 16 : NS_USED;
    // values MMA columns: one per head (INT4: per (group, head))
    static constexpr int NO_USED = INT4 ? NGR * G : G;
    static constexpr int NO = NO_USED <= 16 ? 16 : NO_USED;
    static_assert(NS % 16 == 0 && NS <= 256 && NO % 16 == 0 && NO <= 256, "M = 128 MMA needs N % 16 == 0");
    // tensor memory columns
    static constexpr int KCOL = D / 2;  // fp16 pairs of one K row
    static constexpr int TM_K = 0;      // 2 x KCOL
    // KCH: the low parts of the K rows, 2 x KCOL more (code * factor = hi + lo
    // exactly; the scores MMA accumulates both)
    static constexpr int TM_KLO = 2 * KCOL;
    static constexpr int TM_S = (KCH ? 4 : 2) * KCOL;
    static constexpr int TM_O = TM_S + 2 * NS;
    static constexpr int TM_USED = TM_O + 2 * NO;
    static constexpr int TM_COLS = TM_USED <= 32 ? 32 : TM_USED <= 64 ? 64 : TM_USED <= 128 ? 128
                                 : TM_USED <= 256 ? 256 : 512;
    static_assert(TM_USED <= 512, "tensor memory");
    // threads: token group 0-3, channel group 4-7, NPW producer warps, the MMA warp
    // producer warps (measured: INT8 and per-channel K gain from a fourth,
    // FP8 loses with it; symmetric INT4 stays at three for registers)
    static constexpr int NPW = INT8 ? 4 : 3;
    static constexpr int PR_WARP0 = 8, MM_WARP = PR_WARP0 + NPW;
    static constexpr int THREADS = 32 * (MM_WARP + 1);
    // one raw stage (bytes)
    static constexpr int RK = 0;
    static constexpr int RV = RK + T * CB;
    static constexpr int RKS = RV + T * CB;
    static constexpr int RVS = RKS + T * MB;
    static constexpr int RKZ = RVS + T * MB;
    static constexpr int RVZ = RKZ + (INT4 && !SYM4 ? T * MB : 0);
    static constexpr int RQ = RVZ + (INT4 && !SYM4 ? T * MB : 0);
    static constexpr int RKC = RQ + G * D * 2;             // per unit: D fp16 channel factors (KCH)
    static constexpr int STAGE = RKC + (KCH ? TU * D * 2 : 0);
    // operand buffers: V^T (128 channel rows x T tokens, fp16, MN-major:
    // (c, t) at (c/8)*VS_SBO + (t/8)*128 + (t%8)*16 + (c%8)*2), the query
    // operand (NS rows x D, K-major: (n, c) at (n/8)*QB_SBO + (c/8)*128 +
    // (n%8)*16 + (c%8)*2) and the weights (T tokens x NO, MN-major:
    // (t, n) at (n/8)*WB_SBO + (t/8)*128 + (t%8)*16 + (n%8)*2)
    static constexpr int VS_SBO = (T / 8) * 128;
    static constexpr int VS_BYTES = 16 * VS_SBO;  // 128 rows: rows >= D are zero
    static constexpr int QB_SBO = (D / 8) * 128;
    static constexpr int QB_BYTES = (NS / 8) * QB_SBO;
    static constexpr int WB_SBO = (T / 8) * 128;
    static constexpr int WB_BYTES = (NO / 8) * WB_SBO;
    // small per-tile / per-piece state
    static constexpr int PINFO = 2 * G + (INT4 ? NGR * G : 0);  // L[G], M[G], Z[G][NGR]
    static constexpr int PSC = G + (INT4 ? 2 * NGR * G : 0);    // sq[G], bsum hi/lo [G][NGR] (as float)
    static constexpr int NBAR_FIXED = 15;                       // 7 pairs + drain
    // layout
    static constexpr int OFF_VS = 0;
    static constexpr int OFF_QB = OFF_VS + 2 * VS_BYTES;
    static constexpr int OFF_WB = OFF_QB + 2 * QB_BYTES;
    static constexpr int OFF_SMALL = OFF_WB + 2 * WB_BYTES;
    static constexpr int SMALL_BYTES = 16                   // tmem base, abort flag, misc
                                       + 8 * 2              // plan scratch (int64)
                                       + 4 * 8              // stage bad masks (up to 8 stages)
                                       + 4 * 2 * 4 * (G + 1)  // tile max keys [2][4 warps][G + 1]
                                       + 4 * 2 * (G + 1)      // tile info [2][alpha[G], vsmax]
                                       + 4 * 2 * PINFO        // piece results [2]
                                       + 4 * 2 * PSC          // piece scalars [2]
                                       + 4 * 4 * PINFO;       // piece reduction scratch [4 warps]
    static constexpr int OFF_RAW0 = (OFF_SMALL + SMALL_BYTES + 127) / 128 * 128;
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int PREFIX_MAX = (MAX_SEQS + 1) * 4;
    static constexpr int STATIC_SLACK = 2048;  // the kernel's static shared memory (plan scan, merge list)
    static constexpr int R_FIT = (SMEM_LIMIT - STATIC_SLACK - OFF_RAW0 - PREFIX_MAX - 8 * (NBAR_FIXED + 16)) / STAGE;
    static constexpr int R = R_FIT > 6 ? 6 : R_FIT;  // raw stages
    static_assert(R >= 2, "at least two raw stages");
    static constexpr int OFF_BAR = OFF_RAW0 + R * STAGE;
    static constexpr int NBAR = 2 * R + NBAR_FIXED;
    static constexpr int OFF_PREFIX = OFF_BAR + 8 * NBAR;
    static size_t smem_bytes(int B) { return (size_t)OFF_PREFIX + (size_t)(B + 1) * 4; }
    static_assert(STAGE % 16 == 0 && OFF_RAW0 % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
    static_assert((UNIT * MB) % 16 == 0 && (G * D * 2) % 16 == 0, "16-byte copies");
};

// Offsets of the small state inside the OFF_SMALL region.
template <class C, int G>
struct Small {
    uint8_t* base;
    __device__ uint32_t* tmem_base() const { return reinterpret_cast<uint32_t*>(base); }
    __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + 4); }
    __device__ int64_t* plan_misc() const { return reinterpret_cast<int64_t*>(base + 16); }
    __device__ uint32_t* stage_bad() const { return reinterpret_cast<uint32_t*>(base + 32); }
    __device__ int* red(int buf) const { return reinterpret_cast<int*>(base + 64) + buf * 4 * (G + 1); }
    __device__ float* info(int buf) const {
        return reinterpret_cast<float*>(base + 64 + 4 * 2 * 4 * (G + 1)) + buf * (G + 1);
    }
    __device__ float* pinfo(int buf) const {
        return reinterpret_cast<float*>(base + 64 + 4 * 2 * 4 * (G + 1) + 4 * 2 * (G + 1)) + buf * C::PINFO;
    }
    __device__ float* psc(int buf) const {
        return reinterpret_cast<float*>(base + 64 + 4 * 2 * 4 * (G + 1) + 4 * 2 * (G + 1) + 4 * 2 * C::PINFO) +
               buf * C::PSC;
    }
    __device__ float* pred(int warp) const {
        return reinterpret_cast<float*>(base + 64 + 4 * 2 * 4 * (G + 1) + 4 * 2 * (G + 1) + 4 * 2 * C::PINFO +
                                        4 * 2 * C::PSC) +
               warp * C::PINFO;
    }
};

// The tiles of a CTA's slice, piece by piece: tile = up to TU units of one
// piece, starting at unit u0 of the segment.
struct TileIter {
    PieceWalk w;
    Piece pc;
    int u0;
    int piece;  // index of the current piece in this CTA's slice
    bool valid;
    __device__ void seek(const DecodeParams& p) {
        while (!w.done()) {
            pc = w.get(p);
            if (pc.u_lo < pc.u_hi) {
                u0 = pc.u_lo;
                ++piece;
                valid = true;
                return;
            }
            w.next();
        }
        valid = false;
    }
    __device__ void begin(const Plan& pl, const int32_t* prefix, const DecodeParams& p) {
        w.begin(pl, prefix, blockIdx.x, pl.S);
        piece = -1;
        valid = false;
        seek(p);
    }
    template <int TU>
    __device__ void next(const DecodeParams& p) {
        u0 += TU;
        if (u0 >= pc.u_hi) {
            w.next();
            seek(p);
        }
    }
    __device__ bool first() const { return u0 == pc.u_lo; }
    template <int TU>
    __device__ bool last() const { return u0 + TU >= pc.u_hi; }
    template <int TU>
    __device__ int nunits() const { return min(TU, pc.u_hi - u0); }
};

// ---------------------------------------------------------------- the kernel
template <int SCHEME, int D, int G>
__global__ void __launch_bounds__(Cfg<SCHEME, D, G>::THREADS, 1) decode_tc_kernel(const DecodeParams p) {
    using C = Cfg<SCHEME, D, G>;
    constexpr int T = C::T, TU = C::TU, R = C::R;
    extern __shared__ __align__(128) uint8_t smem[];
    // Launched with programmatic stream serialization: the CTAs may be
    // resident before the kernel ahead of them in the stream ends.  The
    // set-up that uses no array behind a pointer (barriers, tensor memory,
    // zeroing shared memory) runs at once; lengths, tables, queries, cache
    // and workspace are touched only after the wait, once that kernel has
    // completed and its writes are visible.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Small<C, G> sm{smem + C::OFF_SMALL};
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + C::OFF_PREFIX);
    const uint32_t bar0 = smem_addr(smem + C::OFF_BAR);
    // barrier addresses
    auto full = [&](int s) { return bar0 + 8 * s; };
    auto empty = [&](int s) { return bar0 + 8 * (R + s); };
    auto kready = [&](int b) { return bar0 + 8 * (2 * R + 0 + b); };
    auto vready = [&](int b) { return bar0 + 8 * (2 * R + 2 + b); };
    auto wready = [&](int b) { return bar0 + 8 * (2 * R + 4 + b); };
    auto sdone = [&](int b) { return bar0 + 8 * (2 * R + 6 + b); };
    auto odone = [&](int b) { return bar0 + 8 * (2 * R + 8 + b); };
    auto accdone = [&](int b) { return bar0 + 8 * (2 * R + 10 + b); };
    auto pready = [&](int b) { return bar0 + 8 * (2 * R + 12 + b); };
    const uint32_t drain = bar0 + 8 * (2 * R + 14);

    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(full(s), C::NPW * (32 + 1));  // per producer warp: 32 lanes' copies + its lane 0
            mbar_init(empty(s), 8);      // 4 token warps + 4 channel warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(kready(b), 4);
            mbar_init(vready(b), 4);
            mbar_init(wready(b), 4);
            mbar_init(sdone(b), 1);
            mbar_init(odone(b), 1);
            mbar_init(accdone(b), 4);
            mbar_init(pready(b), 1);
        }
        mbar_init(drain, 1);
        *sm.abort_flag() = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == C::MM_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(sm.tmem_base())),
                     "n"(C::TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // zero the operand buffers' constant parts: V^T rows >= D, query rows
    // and blocks never written, weight columns >= NO_USED
    for (int i = tid; i < (2 * C::VS_BYTES + 2 * C::QB_BYTES + 2 * C::WB_BYTES) / 16; i += C::THREADS)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    grid_dependency_wait();  // the kernel ahead has completed
    const Plan plan = build_plan<C::THREADS>(p, prefix, sm.plan_misc());  // contains __syncthreads
    if (blockIdx.x == 0) {
        // publish the plan for the merge kernel: [U, S] then prefix[0..B]
        int64_t* wsplan = reinterpret_cast<int64_t*>(p.ws_l + 2 * (size_t)p.n_ctas * G);
        if (tid == 0) {
            wsplan[0] = plan.U;
            wsplan[1] = plan.S;
        }
        int32_t* wp = reinterpret_cast<int32_t*>(wsplan + 2);
        for (int b = tid; b <= p.B; b += C::THREADS) wp[b] = prefix[b];
    }
    if (p.fuse_merge) {  // empty sequences get zero rows (no CTA's slice touches them)
        for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
            if (prefix[b + 1] != prefix[b]) continue;
            const OutRow row = out_row(p, (int64_t)b * p.Hq * D);
            for (int i = tid; i < p.Hq * D; i += C::THREADS) store_out(row, i, 0.0f);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_base();
    const int Hkv = p.c.num_kv_heads;
    const int P = p.c.page_size;

    if (warp >= C::PR_WARP0 && warp < C::PR_WARP0 + C::NPW) {
        // ------------------------------------------------------------ producers
        // NPW warps fill each stage together: warp pw copies units pw, pw +
        // NPW, ... of the tile (a single warp's 16-byte copies cannot keep up
        // with the consumers); the last warp also copies a piece's query rows.
        const int pw = warp - C::PR_WARP0;
        TileIter it;
        it.begin(plan, prefix, p);
        // page id of this lane's unit of tile t2 (lane < units of the tile),
        // loaded one tile ahead of its copies
        auto page_of = [&](const TileIter& t2) -> int {
            if (!t2.valid || lane >= t2.template nunits<TU>()) return -1;
            const int lp = ((t2.u0 + lane) * UNIT) / P;
            return __ldg(p.block_table + (int64_t)t2.pc.b * p.max_pages + lp);
        };
        int my_page = page_of(it);
        for (int i = 0; it.valid; ++i) {
            const int s = i % R;
            if (i >= R && !mbar_wait(empty(s), ((i / R) - 1) & 1, p.err)) {
                *sm.abort_flag() = 1;
                break;
            }
            if (*sm.abort_flag()) break;
            TileIter nx = it;
            nx.template next<TU>(p);
            const int next_page = page_of(nx);
            uint8_t* st = smem + C::OFF_RAW0 + s * C::STAGE;
            const Piece& pc = it.pc;
            const int nu = it.template nunits<TU>();
            if (it.first() && pw == C::NPW - 1) {  // the piece's query rows travel with its first tile
                const uint8_t* qsrc =
                    reinterpret_cast<const uint8_t*>(p.q + ((int64_t)pc.b * p.Hq + (int64_t)pc.h * G) * D);
                constexpr int NQ = G * D * 2 / 16;
                for (int c = lane; c < NQ; c += 32) cp_async16(st + C::RQ + 16 * c, qsrc + 16 * c);
            }
            // units whose page id lies outside the pool are not copied (every
            // warp sees the whole mask; warp 0 publishes it)
            const uint32_t bad =
                __ballot_sync(0xffffffffu, lane < nu && (my_page < 0 || my_page >= p.c.num_pages + p.c.host_pages));
            for (int uu = pw; uu < nu; uu += C::NPW) {
                const int page = __shfl_sync(0xffffffffu, my_page, uu);
                if ((bad >> uu) & 1u) continue;
                const int u = it.u0 + uu;
                const int off = u * UNIT - ((u * UNIT) / P) * P;
                const PagePools pp = page_pools(p.c, page);  // the page's tier (warp-uniform)
                const int64_t row = ((int64_t)pp.index * Hkv + pc.h) * P + off;
                const uint8_t* kc = pp.k_codes + row * C::CB;
                const uint8_t* vc = pp.v_codes + row * C::CB;
                constexpr int NC = UNIT * C::NCH;  // 16-byte chunks of one unit's codes
#pragma unroll
                for (int k = 0; k < (NC + 31) / 32; ++k) {
                    const int c = k * 32 + lane;
                    if (NC % 32 == 0 || c < NC) {
                        const int L = uu * NC + c;  // chunk index within the tile (row-major)
                        cp_async16(st + C::RK + 16 * swz(L), kc + 16 * c);
                        cp_async16(st + C::RV + 16 * swz(L), vc + 16 * c);
                    }
                }
                constexpr int NS16 = UNIT * C::MB / 16;  // 16-byte chunks of one scale (or zero) run
                const int which = lane / NS16, part = lane % NS16;
                const uint8_t* src = nullptr;
                int dst = 0;
                if (which == 0) { src = pp.k_scales; dst = C::RKS; }
                else if (which == 1) { src = pp.v_scales; dst = C::RVS; }
                else if (C::INT4 && !C::SYM4 && which == 2) { src = pp.k_zeros; dst = C::RKZ; }
                else if (C::INT4 && !C::SYM4 && which == 3) { src = pp.v_zeros; dst = C::RVZ; }
                if (src) cp_async16(st + dst + uu * UNIT * C::MB + 16 * part, src + row * C::MB + 16 * part);
                if constexpr (C::KCH) {  // the unit's page's channel factors: lanes 16 .. 16 + D/8 - 1
                    const int cl = lane - 16;
                    if (cl >= 0 && cl < D / 8)
                        cp_async16(st + C::RKC + uu * D * 2 + 16 * cl,
                                   pp.k_chan + ((int64_t)pp.index * Hkv + pc.h) * D * 2 + 16 * cl);
                }
            }
            if (pw == 0 && lane == 0) {
                sm.stage_bad()[s] = bad;
                if (bad) flag_error(p.err, ERR_BAD_TABLE);
            }
            __syncwarp();
            cp_async_arrive_noinc(full(s));
            if (lane == 0) mbar_arrive(full(s));
            my_page = next_page;
            it = nx;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == C::MM_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDS = idesc_f16(128, C::NS, 0, 0);
            constexpr uint32_t IDO = idesc_f16(128, C::NO, 1, 1);
            const uint32_t qb0 = smem_addr(smem + C::OFF_QB), vs0 = smem_addr(smem + C::OFF_VS),
                           wb0 = smem_addr(smem + C::OFF_WB);
            TileIter it;
            it.begin(plan, prefix, p);
            int i = 0;
            bool ok = true;
            auto issue_values = [&](int j) {
                const int b = j & 1;
                if (!mbar_wait(vready(b), (j >> 1) & 1, p.err) || !mbar_wait(wready(b), (j >> 1) & 1, p.err)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t a = vs0 + b * C::VS_BYTES, w = wb0 + b * C::WB_BYTES;
#pragma unroll
                for (int kk = 0; kk < T / 16; ++kk)
                    mma_smem_a(tmem + C::TM_O + b * C::NO, smem_desc(a + kk * 256, 128, C::VS_SBO),
                               smem_desc(w + kk * 256, 128, C::WB_SBO), IDO, kk > 0);
                mma_commit(odone(b));
            };
            for (; it.valid && ok; it.template next<TU>(p), ++i) {
                const int b = i & 1;
                if (!mbar_wait(kready(b), (i >> 1) & 1, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t q = qb0 + (it.piece & 1) * C::QB_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_tmem_a(tmem + C::TM_S + b * C::NS, tmem + C::TM_K + b * C::KCOL + kk * 8,
                               smem_desc(q + kk * 256, 128, C::QB_SBO), IDS, kk > 0);
                if constexpr (C::KCH) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_tmem_a(tmem + C::TM_S + b * C::NS, tmem + C::TM_KLO + b * C::KCOL + kk * 8,
                                   smem_desc(q + kk * 256, 128, C::QB_SBO), IDS, true);
                }
                mma_commit(sdone(b));
                if (i >= 1) issue_values(i - 1);
            }
            if (ok && i >= 1) issue_values(i - 1);
            if (!ok) *sm.abort_flag() = 1;
            // drain: every MMA issued above has completed once this commit arrives
            mma_commit(drain);
            mbar_wait(drain, 0, p.err);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ token group
        const int t = tid;  // token of the tile = tensor-memory lane
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        float m_run[G], l_part[G];
        float zacc[G][C::INT4 ? C::NGR : 1];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_part[g] = 0.0f;
#pragma unroll
            for (int r = 0; r < (C::INT4 ? C::NGR : 1); ++r) zacc[g][r] = 0.0f;
        }
        // per-token scales of the tile being widened (nxt) and of the tile in softmax (cur)
        constexpr int NSC = C::INT4 ? C::NGR : 1;
        float ks_c[NSC], vs_c[NSC], kz_c[NSC], vz_c[NSC];
        float ks_n[NSC], vs_n[NSC], kz_n[NSC], vz_n[NSC];
        bool valid_c = false, valid_n = false;
        bool bad = false;

        // Widens tile j's K codes of token t into tensor memory (and, at a
        // piece's first tile, builds the query operand and its scalars).
        auto widen = [&](const TileIter& it, int j) {
            const int s = j % R;
            if (!mbar_wait(full(s), (j / R) & 1, p.err)) {
                bad = true;
                return;
            }
            const uint8_t* st = smem + C::OFF_RAW0 + s * C::STAGE;
            const uint32_t badm = sm.stage_bad()[s];
            const int nu = it.template nunits<TU>();
            const int uu = t / UNIT;
            valid_n = uu < nu && !((badm >> uu) & 1u) && (it.u0 + uu) * UNIT + (t % UNIT) < it.pc.len;
            if (it.first()) {
                // query operand of the piece: thread (g, 8-channel block); every
                // thread of the group takes part in the shuffles
                constexpr int TPH = D / 8;
                const int pb = it.piece & 1;
                uint8_t* qb = smem + C::OFF_QB + pb * C::QB_BYTES;
                float* psc = sm.psc(pb);
                const bool qa = t < G * TPH;
                const int g = qa ? t / TPH : 0, blk = t % TPH;
                float qf[8];
                {
                    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                    if (qa) raw = *reinterpret_cast<const uint4*>(st + C::RQ + (g * D + blk * 8) * 2);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        qf[2 * k] = bf16_bits_to_float(w4[k] & 0xFFFFu);
                        qf[2 * k + 1] = bf16_bits_to_float(w4[k] >> 16);
                    }
                }
                if constexpr (C::FP8) {
                    uint32_t h[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __half2 x = __floats2half2_rn(qf[2 * k], qf[2 * k + 1]);
                        h[k] = *reinterpret_cast<const uint32_t*>(&x);
                    }
                    if (qa)
                        *reinterpret_cast<uint4*>(qb + (g / 8) * C::QB_SBO + blk * 128 + (g % 8) * 16) =
                            make_uint4(h[0], h[1], h[2], h[3]);
                } else {
                    // 16-bit fixed point per head: q ~ sq (256 hi + lo)
                    float amax = 0.0f;
#pragma unroll
                    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(qf[k]));
#pragma unroll
                    for (int off = TPH / 2; off >= 1; off >>= 1)
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                    const float inv = amax > 0.0f ? 32767.0f / amax : 0.0f;
                    int qi[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) qi[k] = __float2int_rn(qf[k] * inv);
                    // element k of the stored 8-block holds channel blk*8 + perm(k)
                    auto chan = [&](int k) { return C::INT4 ? int4_perm8(k) : k; };
                    uint32_t hw[4], lw[4];
                    int hs = 0, ls = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int a = qi[chan(2 * k)], b2 = qi[chan(2 * k + 1)];
                        const __half2 hh = __floats2half2_rn((float)(a >> 8), (float)(b2 >> 8));
                        const __half2 ll = __floats2half2_rn((float)(a & 255), (float)(b2 & 255));
                        hw[k] = *reinterpret_cast<const uint32_t*>(&hh);
                        lw[k] = *reinterpret_cast<const uint32_t*>(&ll);
                        hs += (a >> 8) + (b2 >> 8);
                        ls += (a & 255) + (b2 & 255);
                    }
                    int nh, nl;
                    if constexpr (C::INT8) {
                        nh = g;
                        nl = G + g;
                    } else {
                        const int grp = blk / 4;  // 32-channel group of this 8-channel block
                        nh = (0 * C::NGR + grp) * G + g;
                        nl = (1 * C::NGR + grp) * G + g;
                    }
                    if (qa) {
                        *reinterpret_cast<uint4*>(qb + (nh / 8) * C::QB_SBO + blk * 128 + (nh % 8) * 16) =
                            make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(qb + (nl / 8) * C::QB_SBO + blk * 128 + (nl % 8) * 16) =
                            make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        if (blk == 0) psc[g] = (amax / 32767.0f) * p.q_scale;
                    }
                    if constexpr (C::INT4) {
                        // group sums of the hi and lo bytes over the 4 blocks of a group
                        hs += __shfl_xor_sync(0xffffffffu, hs, 1);
                        hs += __shfl_xor_sync(0xffffffffu, hs, 2);
                        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
                        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
                        if (qa && blk % 4 == 0) {
                            psc[G + g * C::NGR + blk / 4] = (float)hs;
                            psc[G + G * C::NGR + g * C::NGR + blk / 4] = (float)ls;
                        }
                    }
                }
            }
            // this token's scales
            if constexpr (C::SYM4) {
#pragma unroll
                for (int r = 0; r < C::NGR; ++r) {
                    ks_n[r] = reinterpret_cast<const float*>(st + C::RKS)[t * C::NGR + r];
                    vs_n[r] = reinterpret_cast<const float*>(st + C::RVS)[t * C::NGR + r];
                    kz_n[r] = -8.0f * ks_n[r];  // exact
                    vz_n[r] = -8.0f * vs_n[r];
                }
            } else if constexpr (C::INT4) {
#pragma unroll
                for (int r = 0; r < C::NGR; ++r) {
                    ks_n[r] = __half2float(reinterpret_cast<const __half*>(st + C::RKS)[t * C::NGR + r]);
                    vs_n[r] = __half2float(reinterpret_cast<const __half*>(st + C::RVS)[t * C::NGR + r]);
                    kz_n[r] = __half2float(reinterpret_cast<const __half*>(st + C::RKZ)[t * C::NGR + r]);
                    vz_n[r] = __half2float(reinterpret_cast<const __half*>(st + C::RVZ)[t * C::NGR + r]);
                }
            } else {
                ks_n[0] = reinterpret_cast<const float*>(st + C::RKS)[t];
                vs_n[0] = reinterpret_cast<const float*>(st + C::RVS)[t];
            }
            // widen the K row into tensor memory, 16 columns at a time
            const uint32_t ta = tl + C::TM_K + (j & 1) * C::KCOL;
            constexpr int CPS = C::INT4 ? 1 : 2;  // raw 16-byte chunks per 16 columns
            // kept rolled (as the V widening below): the kernel's four roles
            // run different code, and the smaller body costs fewer
            // instruction-cache misses than the unrolled one saves (FP8,
            // whose conversions are longer, measured best at two per pass)
            constexpr int KUNR = C::FP8 ? 2 : 1;
#pragma unroll KUNR
            for (int c0 = 0; c0 < C::NCH; c0 += CPS) {
                uint32_t r[16];
                uint32_t rlo[C::KCH ? 16 : 1];  // KCH: the low parts
#pragma unroll
                for (int cc = 0; cc < CPS; ++cc) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(st + C::RK + 16 * swz(t * C::NCH + c0 + cc));
                    const uint32_t w4[4] = {raw.x ^ C::NIBX, raw.y ^ C::NIBX, raw.z ^ C::NIBX, raw.w ^ C::NIBX};
                    if constexpr (C::INT8) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) s8x4_to_h2x2(w4[k], r[cc * 8 + 2 * k], r[cc * 8 + 2 * k + 1]);
                        if constexpr (C::KCH) {
                            // r[cc * 8 + i] holds channels 16 (c0 + cc) + 2i, + 1:
                            // times the unit's factors of the same channels as
                            // hi = fp16(code * f) and lo = fp16(code * f - hi),
                            // whose sum is the product exactly (code * f has at
                            // most 18 significant bits on the grid of f's last
                            // bit, so the remainder fits fp16); the token scale
                            // follows the MMA
                            const uint4* f =
                                reinterpret_cast<const uint4*>(st + C::RKC + uu * D * 2 + (c0 + cc) * 32);
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const uint4 fv = f[h2];
                                const uint32_t fw[4] = {fv.x, fv.y, fv.z, fv.w};
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const __half2 x = *reinterpret_cast<const __half2*>(&r[cc * 8 + h2 * 4 + k]);
                                    const __half2 fk = *reinterpret_cast<const __half2*>(&fw[k]);
                                    // hi rounded on its own (__hmul2_rn: never contracted
                                    // into the fma below, which would make lo 0)
                                    const __half2 hi = __hmul2_rn(x, fk);
                                    const __half2 lo = __hfma2(x, fk, __hneg2(hi));
                                    r[cc * 8 + h2 * 4 + k] = *reinterpret_cast<const uint32_t*>(&hi);
                                    rlo[cc * 8 + h2 * 4 + k] = *reinterpret_cast<const uint32_t*>(&lo);
                                }
                            }
                        }
                    } else if constexpr (C::FP8) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            r[cc * 8 + 2 * k] = e4m3x2_to_h2(w4[k]);
                            r[cc * 8 + 2 * k + 1] = e4m3x2_to_h2(w4[k] >> 16);
                        }
                    } else {
                        // 8 nibbles per word -> 4 columns (biased by 1024, removed in the epilogue)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            r[cc * 16 + 4 * k + 0] = nib_pair(w4[k]);
                            r[cc * 16 + 4 * k + 1] = nib_pair(w4[k] >> 4);
                            r[cc * 16 + 4 * k + 2] = nib_pair(w4[k] >> 8);
                            r[cc * 16 + 4 * k + 3] = nib_pair(w4[k] >> 12);
                        }
                    }
                }
                tmem_st16(ta + c0 * (C::INT4 ? 16 : 8), r);
                if constexpr (C::KCH) tmem_st16(ta + (C::TM_KLO - C::TM_K) + c0 * 8, rlo);
            }
            tmem_st_wait();
            fence_proxy_async_smem();  // query operand writes
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(kready(j & 1));
                mbar_arrive(empty(s));
            }
        };

        TileIter it;
        it.begin(plan, prefix, p);
        if (it.valid) widen(it, 0);
        bad = tg_barrier_any(bad);  // also publishes the first piece's scalars
        int i = 0;
        while (it.valid && !bad) {
            TileIter nx = it;
            nx.template next<TU>(p);
#pragma unroll
            for (int r = 0; r < NSC; ++r) {
                ks_c[r] = ks_n[r];
                vs_c[r] = vs_n[r];
                kz_c[r] = kz_n[r];
                vz_c[r] = vz_n[r];
            }
            valid_c = valid_n;
            if (nx.valid) widen(nx, i + 1);
            // ---- softmax of tile i
            const int b = i & 1;
            const int pb = it.piece & 1;
            const float* psc = sm.psc(pb);
            bool ok = mbar_wait(sdone(b), (i >> 1) & 1, p.err);
            if (ok && i >= 2) ok = mbar_wait(accdone(b), ((i - 2) >> 1) & 1, p.err);
            tc_fence_after();
            float s[G];
            if (ok) {
                uint32_t sr[(C::NS_USED + 15) / 16 * 16];
#pragma unroll
                for (int c0 = 0; c0 < C::NS_USED; c0 += 16) tmem_ld16(tl + C::TM_S + b * C::NS + c0, sr + c0);
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v;
                    if constexpr (C::KCH) {
                        // the sums carry fractions (codes times factors): recombined
                        // in fp32, not through integers
                        const float sh = fmaf(__uint_as_float(sr[g]), 256.0f, __uint_as_float(sr[G + g]));
                        v = sh * (psc[g] * ks_c[0]);
                    } else if constexpr (C::INT8) {
                        const int ai = (int)__uint_as_float(sr[g]) * 256 + (int)__uint_as_float(sr[G + g]);
                        v = (float)ai * (psc[g] * ks_c[0]);
                    } else if constexpr (C::FP8) {
                        v = __uint_as_float(sr[g]) * (ks_c[0] * p.q_scale);
                    } else {
                        float acc = 0.0f;
#pragma unroll
                        for (int r = 0; r < C::NGR; ++r) {
                            const int bh = (int)psc[G + g * C::NGR + r], bl = (int)psc[G + G * C::NGR + g * C::NGR + r];
                            const int dh = (int)__uint_as_float(sr[(0 * C::NGR + r) * G + g]) - 1024 * bh;
                            const int dl = (int)__uint_as_float(sr[(1 * C::NGR + r) * G + g]) - 1024 * bl;
                            acc = fmaf(ks_c[r], (float)(dh * 256 + dl), fmaf(kz_c[r], (float)(bh * 256 + bl), acc));
                        }
                        v = acc * psc[g];
                    }
                    s[g] = valid_c ? v : -INFINITY;
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) s[g] = -INFINITY;
            }
            // tile maxima of the scores (per head) and of the value scales
            float vmax_t = 0.0f;
            if (valid_c) {
#pragma unroll
                for (int r = 0; r < NSC; ++r) vmax_t = fmaxf(vmax_t, vs_c[r]);
            }
            int* red = sm.red(b);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int k = __reduce_max_sync(0xffffffffu, fkey(s[g]));
                if (lane == 0) red[warp * (G + 1) + g] = k;
            }
            {
                const int k = __reduce_max_sync(0xffffffffu, __float_as_int(vmax_t));  // non-negative
                if (lane == 0) red[warp * (G + 1) + G] = k;
            }
            bad = tg_barrier_any(!ok || bad);
            if (bad) break;
            float mt[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                int k = red[g];
#pragma unroll
                for (int w2 = 1; w2 < 4; ++w2) k = max(k, red[w2 * (G + 1) + g]);
                mt[g] = fkey_inv(k);
            }
            int kv = red[G];
#pragma unroll
            for (int w2 = 1; w2 < 4; ++w2) kv = max(kv, red[w2 * (G + 1) + G]);
            const float vsmax = __int_as_float(kv);
            const float inv_vs = vsmax > 0.0f ? 1.0f / vsmax : 0.0f;
            float alpha[G];
            float wv[C::NO_USED];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float m_new = fmaxf(m_run[g], mt[g]);
                alpha[g] = (m_run[g] == -INFINITY) ? 0.0f : fast_exp2(m_run[g] - m_new);
                const float pr = (s[g] == -INFINITY) ? 0.0f : fast_exp2(s[g] - m_new);
                m_run[g] = m_new;
                l_part[g] = fmaf(l_part[g], alpha[g], pr);
                // masked tokens: p = 0, and their scales are not read (may be garbage)
                if constexpr (C::INT4) {
#pragma unroll
                    for (int r = 0; r < C::NGR; ++r) {
                        zacc[g][r] = valid_c ? fmaf(zacc[g][r], alpha[g], pr * vz_c[r]) : zacc[g][r] * alpha[g];
                        wv[r * G + g] = valid_c ? pr * (vs_c[r] * inv_vs) : 0.0f;
                    }
                } else {
                    wv[g] = valid_c ? pr * (vs_c[0] * inv_vs) : 0.0f;
                }
            }
            // the weights W[t][n] (MN-major: 8 columns of token t per 16 bytes)
            uint8_t* wb = smem + C::OFF_WB + b * C::WB_BYTES;
#pragma unroll
            for (int n0 = 0; n0 < C::NO_USED; n0 += 8) {
                uint32_t h[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = (n0 + 2 * k < C::NO_USED) ? wv[n0 + 2 * k] : 0.0f;
                    const float c2 = (n0 + 2 * k + 1 < C::NO_USED) ? wv[n0 + 2 * k + 1] : 0.0f;
                    const __half2 x = __floats2half2_rn(a, c2);
                    h[k] = *reinterpret_cast<const uint32_t*>(&x);
                }
                *reinterpret_cast<uint4*>(wb + (n0 / 8) * C::WB_SBO + (t / 8) * 128 + (t % 8) * 16) =
                    make_uint4(h[0], h[1], h[2], h[3]);
            }
            if (t == 0) {
                float* inf = sm.info(b);
#pragma unroll
                for (int g = 0; g < G; ++g) inf[g] = alpha[g];
                inf[G] = vsmax;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(wready(b));
            // ---- end of a piece: the sums over the tile's tokens
            if (it.template last<TU>()) {
                float* pr = sm.pred(warp);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = l_part[g];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == 0) pr[g] = v;
                    if constexpr (C::INT4) {
#pragma unroll
                        for (int r = 0; r < C::NGR; ++r) {
                            float z = zacc[g][r];
#pragma unroll
                            for (int off = 16; off >= 1; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                            if (lane == 0) pr[2 * G + g * C::NGR + r] = z;
                        }
                    }
                }
                tg_barrier();
                if (t == 0) {
                    float* pi = sm.pinfo(pb);
                    for (int k = 0; k < C::PINFO; ++k) {
                        if (k >= G && k < 2 * G) {
                            pi[k] = m_run[k - G];
                            continue;
                        }
                        float v = 0.0f;
                        for (int w2 = 0; w2 < 4; ++w2) v += sm.pred(w2)[k];
                        pi[k] = v;
                    }
                    mbar_arrive(pready(pb));
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_part[g] = 0.0f;
#pragma unroll
                    for (int r = 0; r < (C::INT4 ? C::NGR : 1); ++r) zacc[g][r] = 0.0f;
                }
            }
            it = nx;
            ++i;
        }
        if (bad) *sm.abort_flag() = 1;
    } else {
        // ------------------------------------------------------------ channel group
        const int ct = tid - 128;  // token for widening V; tensor-memory lane (channel row) for the values
        const int cw = warp - 4;
        const uint32_t tl = tmem + ((uint32_t)(cw * 32) << 16);
        // output channel of tensor-memory row ct (INT4 stores its pairs permuted)
        const int ch = C::INT4 ? (ct & ~7) + int4_perm8(ct & 7) : ct;
        const int grp = ct / 32;  // INT4 group of that channel (rows keep their 32-blocks)
        float o[G];
#pragma unroll
        for (int g = 0; g < G; ++g) o[g] = 0.0f;
        bool bad = false;

        auto widen_v = [&](const TileIter& it, int j) {
            const int s = j % R;
            if (!mbar_wait(full(s), (j / R) & 1, p.err)) {
                bad = true;
                return;
            }
            const uint8_t* st = smem + C::OFF_RAW0 + s * C::STAGE;
            const uint32_t badm = sm.stage_bad()[s];
            const int nu = it.template nunits<TU>();
            const int uu = ct / UNIT;
            const bool valid = uu < nu && !((badm >> uu) & 1u) && (it.u0 + uu) * UNIT + (ct % UNIT) < it.pc.len;
            uint8_t* vs = smem + C::OFF_VS + (j & 1) * C::VS_BYTES + (ct / 8) * 128 + (ct % 8) * 16;
            // the row of a token past the piece (or of a page outside the
            // pool) needs no zeroing where every widened code is finite (INT8,
            // both INT4): its weight is exactly 0.  E4M3 stale bytes can be
            // NaN codes, so FP8 rows are zeroed.
            const bool keep = valid || !C::FP8;
#pragma unroll 1
            for (int c = 0; c < C::NCH; ++c) {
                const uint4 raw = *reinterpret_cast<const uint4*>(st + C::RV + 16 * swz(ct * C::NCH + c));
                const uint32_t w4[4] = {raw.x ^ C::NIBX, raw.y ^ C::NIBX, raw.z ^ C::NIBX, raw.w ^ C::NIBX};
                if constexpr (C::INT4) {
                    // 32 channels (one group): 4 blocks of 8
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t h[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t x = nib_pair(w4[k] >> (4 * e));
                            const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&x),
                                                      __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
                            h[e] = *reinterpret_cast<const uint32_t*>(&y);
                        }
                        const int blk = c * 4 + k;
                        *reinterpret_cast<uint4*>(vs + blk * C::VS_SBO) =
                            keep ? make_uint4(h[0], h[1], h[2], h[3]) : make_uint4(0u, 0u, 0u, 0u);
                    }
                } else {
                    uint32_t h[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if constexpr (C::INT8) {
                            s8x4_to_h2x2(w4[k], h[2 * k], h[2 * k + 1]);
                        } else {
                            h[2 * k] = e4m3x2_to_h2(w4[k]);
                            h[2 * k + 1] = e4m3x2_to_h2(w4[k] >> 16);
                        }
                    }
                    *reinterpret_cast<uint4*>(vs + (2 * c) * C::VS_SBO) =
                        keep ? make_uint4(h[0], h[1], h[2], h[3]) : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(vs + (2 * c + 1) * C::VS_SBO) =
                        keep ? make_uint4(h[4], h[5], h[6], h[7]) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(vready(j & 1));
                mbar_arrive(empty(s));
            }
        };

        TileIter it;
        it.begin(plan, prefix, p);
        if (it.valid) widen_v(it, 0);
        int i = 0;
        while (it.valid && !bad && !*sm.abort_flag()) {
            TileIter nx = it;
            nx.template next<TU>(p);
            if (nx.valid) widen_v(nx, i + 1);
            const int b = i & 1;
            if (bad || !mbar_wait(odone(b), (i >> 1) & 1, p.err) || !mbar_wait(wready(b), (i >> 1) & 1, p.err)) {
                bad = true;
                break;
            }
            tc_fence_after();
            uint32_t dr[8];
            if constexpr (G >= 8) tmem_ld8(tl + C::TM_O + b * C::NO + (C::INT4 ? grp * G : 0), dr);
            else tmem_ld4(tl + C::TM_O + b * C::NO + (C::INT4 ? grp * G : 0), dr);
            tmem_ld_wait();
            const float* inf = sm.info(b);
            const float vsmax = inf[G];
#pragma unroll
            for (int g = 0; g < G; ++g) o[g] = fmaf(o[g], inf[g], __uint_as_float(dr[g]) * vsmax);
            if (it.template last<TU>()) {
                const int pb = it.piece & 1;
                if (!mbar_wait(pready(pb), (it.piece >> 1) & 1, p.err)) {
                    bad = true;
                    break;
                }
                const float* pi = sm.pinfo(pb);
                const Piece& pc = it.pc;
                if (pc.whole) {
                    const OutRow row = out_row(p, ((int64_t)pc.b * p.Hq + (int64_t)pc.h * G) * D);
                    if (ct < D) {
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float L = pi[g];
                            const float z = C::INT4 ? pi[2 * G + g * C::NGR + grp] : 0.0f;
                            store_out(row, g * D + ch, (L > 0.0f) ? (o[g] + z) / L : 0.0f);
                        }
                    }
                } else {
                    const int64_t slot = pc.slot;
                    if (ct < D) {
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float z = C::INT4 ? pi[2 * G + g * C::NGR + grp] : 0.0f;
                            p.ws_o[(slot * G + g) * D + ch] = o[g] + z;
                        }
                    }
                    if (ct < G) {
                        p.ws_m[slot * G + ct] = pi[G + ct];
                        p.ws_l[slot * G + ct] = pi[ct];
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) o[g] = 0.0f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accdone(b));
            it = nx;
            ++i;
        }
        if (bad) *sm.abort_flag() = 1;
    }

    // ---------------------------------------------------------------- exit
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::MM_WARP)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::TM_COLS)
                     : "memory");
    if (*sm.abort_flag() || !p.fuse_merge) return;

    // ---- cross-CTA merge: count this CTA's arrival on the (at most two)
    // segments it shares with other CTAs; merge those it brought last
    __threadfence();
    __syncthreads();
    __shared__ int s_merge[2][4];  // per end piece: b, h, a (work-line start), units; b < 0: nothing
    if (tid < 2) {
        s_merge[tid][0] = -1;
        PieceWalk w;
        w.begin(plan, prefix, blockIdx.x, plan.S);
        // piece 0 (tid 0) or the last piece (tid 1), if it is not whole and not the same piece
        int idx = 0;
        Piece pc{}, first{}, lastp{};
        bool have = false;
        for (; !w.done(); w.next(), ++idx) {
            pc = w.get(p);
            if (idx == 0) first = pc;
            lastp = pc;
            have = true;
        }
        const Piece& e = tid == 0 ? first : lastp;
        if (have && !e.whole && !(tid == 1 && idx == 1)) {
            const int units = prefix[e.b + 1] - prefix[e.b];
            const int64_t a = (int64_t)Hkv * prefix[e.b] + (int64_t)e.h * units;
            const unsigned long long n =
                (unsigned long long)(div_line(a + units - 1, plan.S) - div_line(a, plan.S) + 1);
            if (count_arrival(p, e.b, e.h, n)) {
                s_merge[tid][0] = e.b;
                s_merge[tid][1] = e.h;
                s_merge[tid][2] = (int)(a - div_line(a, plan.S) * plan.S);  // offset of the start in its slice
                s_merge[tid][3] = units;
            }
        }
    }
    __syncthreads();
    __threadfence();  // see the other CTAs' partials
    constexpr int NE = G * D / 4;  // float4 elements of one segment's G output rows
    for (int e = 0; e < 2; ++e) {
        if (s_merge[e][0] < 0) continue;
        const int b = s_merge[e][0], h = s_merge[e][1], units = s_merge[e][3];
        const int64_t a = (int64_t)Hkv * prefix[b] + (int64_t)h * units;
        const int64_t k0 = div_line(a, plan.S), n = div_line(a + units - 1, plan.S) - k0 + 1;
        for (int i0 = warp * 32; i0 < NE; i0 += C::THREADS) {  // warp-uniform trip count
            const int it = i0 + lane;
            merge_element<D, G>(p.ws_o, p.ws_m, p.ws_l, a, plan.S, k0, (int)n, (it % NE) / (D / 4),
                                ((it % NE) % (D / 4)) * 4, lane, it < NE,
                                out_row(p, ((int64_t)b * p.Hq + (int64_t)h * G) * D), nullptr, nullptr, nullptr);
        }
    }
}

// ---------------------------------------------------------------- host side
// Shared memory attribute per device, set once.  Safe to call from several
// host threads: the attribute call is idempotent, and the flag only records
// that it succeeded.
template <int SCHEME, int D, int G>
cudaError_t configure_t() {
    using C = Cfg<SCHEME, D, G>;
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(decode_tc_kernel<SCHEME, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::smem_bytes(MAX_SEQS));
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    return cudaSuccess;
}

// Resident CTAs per SM (the persistent grid is this times the SM count),
// taken at the largest shared-memory size any batch needs; queried once per
// device and cached (a failed query is not cached).
template <int SCHEME, int D, int G>
int ctas_per_sm_t() {
    using C = Cfg<SCHEME, D, G>;
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
    if (configure_t<SCHEME, D, G>() != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tc_kernel<SCHEME, D, G>, C::THREADS,
                                                      C::smem_bytes(MAX_SEQS)) != cudaSuccess)
        return 0;
    if (n > 1) n = 1;  // one CTA per SM: the tensor memory is allocated whole
    if (n > 0) cached[dev].store(n, std::memory_order_release);
    return n;
}

template <int SCHEME, int D, int G>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
    using C = Cfg<SCHEME, D, G>;
    cudaError_t e = configure_t<SCHEME, D, G>();
    if (e != cudaSuccess) return e;
    // programmatic stream serialization: the grid may be scheduled while the
    // kernel ahead of it (typically the append) runs; it waits for it in-kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_ctas);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::smem_bytes(p.B);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<SCHEME, D, G>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int SCHEME>
cudaError_t launch_scheme(const DecodeParams& p, int G_, cudaStream_t s) {
    KVQ_DISPATCH_DG(p.c.head_dim, G_, return (launch_t<SCHEME, D, G>(p, s)));
    return cudaErrorInvalidValue;
}

template <int SCHEME>
int ctas_per_sm_scheme(int head_dim, int G_) {
    KVQ_DISPATCH_DG(head_dim, G_, return (ctas_per_sm_t<SCHEME, D, G>()));
    return 0;
}

}  // namespace tc
}  // namespace kvq
