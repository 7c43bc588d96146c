// kvq_alu.cuh -- split-K fused-dequantization paged GQA decode attention
// (K2) on the CUDA cores, for GQA ratios 1, 2 and 4 of the INT8, FP8 and
// asymmetric INT4 schemes (the tensor-core kernel in kvq_tc.cuh serves GQA 8
// and symmetric INT4; measured on this GPU, each is the faster one where it
// is used).
//
// What it computes ("What is KV Cache Optimization? ...", section "Technical
// Architecture", stage "Fused Dequantization Attention Kernel"; "Dynamic KV
// Cache Quantization for Fast LLM Inference", section "Recap of KV Caching"):
// for sequence b and query head g (KV head h = g / G), softmax over every
// cached token t < seq_len of <q, K_t> / sqrt(d), applied to V_t, where K_t and
// V_t are dequantized from their codes inside the kernel and the pages of the
// sequence are found through its block table.
//
// Decomposition.  The work line of 16-token units (kvq_decode.cuh) is cut
// for a persistent grid of one CTA per SM and WARPS warps each: every warp is
// a worker with its own slice of Sw units, and a CTA's slice (S = WARPS * Sw
// units) is its warps' slices end to end.  A segment that lies inside one
// warp's slice is finished by that warp (final output rows).  Any other piece
// of a warp's slice leaves a warp partial (running max m, sum l, unnormalized
// o) in one of the warp's two slots.  At the end the CTA combines,
// element-parallel, the warp partials of every piece that spans several of
// its warps: a segment that ends inside the CTA's slice gets its final rows,
// one that continues in another CTA gets the CTA's partial (at most two per
// CTA), merged across CTAs as in the tensor-core kernel.
//
// Inside a warp (no producer warp): the warp streams its units through its
// own ring of STAGES shared-memory stages with 16-byte cp.async gathers (all
// 32 lanes issue; page ids come from the block table in 32-entry register
// batches, the next batch prefetched), keeping STAGES-1 units in flight, and
// consumes them:
//  * scores.  INT8: each lane takes ONE query head and D*G/8 of its
//    channels, the query held as 16-bit fixed point (a signed high byte and
//    an unsigned low byte); exact int32 dp4a sums against the codes, summed
//    over the lanes that share the head.  FP8, INT4: each lane holds 16 (or
//    8) channels of all G query rows (INT4 as fixed point with dp4a, FP8 as
//    fp16 with mixed-precision FMAs against exactly converted codes) and a
//    transpose-reduction across the lanes sharing a token leaves one score
//    per lane.  The per-token (and per-head) scales are applied once;
//  * online softmax in base 2 directly on those lanes (max over the unit by
//    shuffles); the weights p * value scale go to shared memory;
//  * values: each lane owns 4 (or 8) channels x G heads of fp32 accumulators.
//    INT8, INT4: the unit's weights of each head (INT4: of each head and
//    32-channel group, since the value scale is per group) become 16-bit
//    fixed point relative to their maximum, packed by the score lanes into
//    words of 4 token bytes; the value lane transposes the codes of the same
//    4 tokens into one word per channel (byte permutes; INT4 masks the two
//    nibbles apart), dp4a accumulates the unit in int32 (high byte, times
//    256, then low byte), and one FMA per accumulator adds the unit.  INT4's
//    zero-point term, sum over tokens of p * zero, is kept per (group, head)
//    on the score lanes and added once when the piece ends.  FP8: scalar
//    FMAs on exactly converted codes.
// The query rows of a piece travel in the stage of the warp's first unit of
// that piece.
#pragma once

#include <atomic>

#include "kvq_decode.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {
namespace alu {

template <int SCHEME, int D, int G>
struct DecodeCfg {
    static constexpr bool INT4 = SCHEME == KVQ_INT4_ASYM_G32;
    static constexpr bool INT8 = SCHEME == KVQ_INT8_SYM_TOKEN;
    // One CTA per SM: with several co-resident CTAs the older CTA's warps win
    // the issue slots and finish first, leaving the SM under-occupied.  INT8
    // fits 128 registers a thread, so 16 warps (with a 2-deep ring each, for
    // shared memory); the others need more registers: 12 warps.
    static constexpr int WARPS = (INT8 || INT4) ? 16 : 12;
    static_assert(WARPS == decode_alu_warps(SCHEME, G), "the workspace is sized for this many warps");
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int CB = INT4 ? D / 2 : D;        // code bytes per token row
    static constexpr int NGR = D / 32;                 // INT4 groups per row
    static constexpr int MB = INT4 ? NGR * 2 : 4;      // bytes per token in one scale/zero array
    static constexpr int Q_BYTES = G * D * 2;          // the query rows of one (sequence, KV head)
    // stage layout (bytes): K codes, V codes, K scales, V scales, [K zeros, V zeros], query rows
    static constexpr int KC = 0;
    static constexpr int VC = KC + UNIT * CB;
    static constexpr int KS = VC + UNIT * CB;
    static constexpr int VS = KS + UNIT * MB;
    static constexpr int KZ = VS + UNIT * MB;
    static constexpr int VZ = KZ + (INT4 ? UNIT * MB : 0);
    static constexpr int QO = VZ + (INT4 ? UNIT * MB : 0);
    static constexpr int STAGE = QO + Q_BYTES;
    // scores: KL lanes per token, CPL channels per lane, TPP tokens per pass.
    // INT8: each lane takes ONE query head (DUP = KL / G lanes per head) and
    // D / DUP of its channels, so its dot product needs no transpose across
    // heads, only a sum over the DUP lanes.  FP8 / INT4: each lane takes 16
    // (or 8) channels of all G heads (INT4: half of one 32-channel scale
    // group) and a transpose-reduction sorts them out.
    static constexpr bool SHEAD = INT8;
    static constexpr int CPL = SHEAD ? D * G / 8 : ((D == 64 && G == 8) ? 8 : 16);
    static constexpr int KL = SHEAD ? 8 : D / CPL;
    static constexpr int QROWS = SHEAD ? 1 : G;  // query rows held per lane
    static constexpr int TPP = 32 / KL;
    static constexpr int PASSES = UNIT / TPP;
    static constexpr int DUP = KL / G;  // lanes that end holding the same (token, head) score
    static constexpr int QW = CPL / 2;  // fp16 pairs of query per head per lane
    static constexpr bool TWO_ACC = G <= 2;  // a second accumulator set for more ILP when registers allow
    // values: VCH channels per lane, VL lanes per token, VT token groups.
    // INT8 and INT4 values go through dp4a: weights as 16-bit fixed point (hi
    // and lo bytes) against the codes of one channel in a block of 4 tokens.
    static constexpr bool VDP = INT8 || INT4;
    static constexpr int VCH = (VDP || (G >= 8 && D == 128)) ? 4 : 8;
    static constexpr int VL = D / VCH;
    static constexpr int VT = 32 / VL;
    static constexpr int V_UNROLL = (G >= 8) ? 4 : UNIT / VT;  // token loop unrolling (register pressure)
    static constexpr int NBLK = UNIT / 4 / VT;                 // dp4a path: 4-token blocks per lane
    // dp4a path: a block is the 4 tokens whose weights LPB score lanes (same
    // channels and head, consecutive token slots) hold over their PASSES
    // passes, so each lane packs its bytes into one store: byte i of block b
    // is token (i % PASSES) * TPP + b * LPB + i / PASSES.
    static constexpr int LPB = 4 / PASSES;
    // INT4 weights carry the value scale of their 32-channel group, so there
    // is one weight per (token, group, head); a score lane computes GPL groups
    static constexpr int NGW = INT4 ? NGR : 1;
    static constexpr int GPL = NGW > DUP ? NGW / DUP : 1;
    // shared memory layout (bytes)
    static constexpr int OFF_STAGES = 0;
    // per warp: weights (fp32 Wt[UNIT][G], or on the dp4a path the words
    // WB[hi, lo][NGW][UNIT/4][G] of 4 token bytes, an order in which the
    // score lanes' stores fall in distinct banks), then the weights'
    // fixed-point step WQ[G] (dp4a path), alpha[G], and (INT4) the
    // zero-point sums ZS[NGR][G] of a finished piece, and the queue of the
    // pieces the feed has reached (b, h, u_lo, u_hi, len, whole, slot, and
    // whether the piece appends its sequence's new token; a negative u_lo
    // ends the list).  The feed runs STAGES - 1 units ahead of
    // the compute and seeks the next piece as it issues a piece's last unit,
    // so it is at most STAGES pieces ahead: 8 slots (STAGES <= 4) never
    // overwrite the compute's current piece.
    static constexpr int NB = UNIT / 4;             // 4-token blocks per unit
    static constexpr int WB_HALF = NGW * NB * G;     // words of one byte plane (hi or lo)
    static constexpr int WB_BYTES = VDP ? 2 * WB_HALF * 4 : UNIT * G * 4;
    static constexpr int W_OFF_WQ = WB_BYTES;
    static constexpr int W_OFF_AL = W_OFF_WQ + G * 4;
    static constexpr int W_OFF_ZS = W_OFF_AL + G * 4;
    static constexpr int W_OFF_PQ = W_OFF_ZS + (INT4 ? NGR * G * 4 : 0);  // piece queue [8][8] int32
    // the appended token's codes, scales (and zeros) as the cache stores them:
    // K codes, V codes [CB], K scales, V scales, K zeros, V zeros [MB]
    static constexpr int W_OFF_NB = (W_OFF_PQ + 8 * 8 * 4 + 15) / 16 * 16;  // 16-byte stores into it
    static constexpr int W_BYTES = (W_OFF_NB + 2 * CB + 4 * MB + 15) / 16 * 16;
    // ring depth per warp (STAGES-1 units in flight): as deep as shared memory
    // allows next to the weights and a plan of MAX_SEQS sequences (227 KB a
    // CTA, less 4 KB for the static arrays), at most 4
    static constexpr int FIT = (232448 - 4096 - WARPS * W_BYTES - 16 - (WARPS + 1) * 48 - (MAX_SEQS + 1) * 4) /
                               (WARPS * STAGE);
    static constexpr int STAGES = FIT < 4 ? FIT : 4;
    static_assert(STAGES >= 2 && STAGES <= 4, "at least one unit in flight while one is computed; the piece queue");
    static constexpr int OFF_W = OFF_STAGES + WARPS * STAGES * STAGE;
    static constexpr int OFF_MISC = OFF_W + WARPS * W_BYTES;
    static constexpr int OFF_EPS = OFF_MISC + 16;  // the CTA's end pieces (EndPiece[WARPS + 1])
    static constexpr int OFF_PLAN = OFF_EPS + (WARPS + 1) * 48;
    static size_t smem_bytes(int B) { return OFF_PLAN + (size_t)(B + 1) * 4; }
    static_assert(G <= KL, "each lane must end the reduction holding one head");
    static_assert(STAGE % 16 == 0 && Q_BYTES % 16 == 0 && (UNIT * MB) % 16 == 0, "16-byte copies");
    static_assert(OFF_W % 16 == 0 && W_BYTES % 16 == 0 && W_OFF_NB % 16 == 0, "alignment");
    static_assert(4 * (UNIT * MB / 16) <= 32, "one lane per 16 bytes of scales and zeros");
    static_assert(!VDP || PASSES == 4 || PASSES == 2, "a lane's weight bytes fill a word or a half word");
    static_assert(!VDP || (NGW % GPL == 0 && NGW / GPL <= DUP), "every group has a writer lane");
    static_assert(!VDP || VCH == 4, "one dp4a word per channel");
};

// Transpose-reduction across the KL lanes that share a token: N values per
// lane in, one (fully summed) value out; the lane ends with head
// (lane % KL) / (KL / G).
template <typename T, int N, int OFF>
__device__ __forceinline__ void transpose_reduce(T* v, int lane) {
    if constexpr (OFF >= 1) {
        if constexpr (N > 1) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const T send = upper ? v[i] : v[i + N / 2];
                const T keep = upper ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            transpose_reduce<T, N / 2, OFF / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            transpose_reduce<T, 1, OFF / 2>(v, lane);
        }
    }
}

// N consecutive fp16 values from shared memory (2N-byte aligned) -> fp32
template <int N>
__device__ __forceinline__ void load_halves(const uint8_t* src, float* f) {
    if constexpr (N == 1) {
        f[0] = __half2float(*reinterpret_cast<const __half*>(src));
    } else {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float2 v = __half22float2(reinterpret_cast<const __half2*>(src)[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
}

struct EndPiece {
    int64_t a;      // work-line unit where the segment starts
    int64_t units;  // units of the segment
    int64_t k0;     // first warp worker touching the piece
    int n;          // warp workers touching it
    int b, h;
    int slot;       // CTA partial slot, or -1: the segment ends here (final rows)
};

// APP: the instantiation of a decode that appends its step's token (kept
// apart so that the plain decode carries none of its registers)
template <int SCHEME, int D, int G, bool APP>
__global__ void __launch_bounds__(DecodeCfg<SCHEME, D, G>::THREADS, 1)
decode_partial_kernel(const DecodeParams p) {
    using C = DecodeCfg<SCHEME, D, G>;
    constexpr int STAGES_ = C::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    // Launched with programmatic stream serialization: the CTAs may be
    // resident before the kernel ahead of them in the stream ends.  Only the
    // kernel's own parameters are used before the wait below; every array
    // behind a pointer (lengths, tables, queries, cache, workspace) is read
    // or written after it, once that kernel has completed and its writes are
    // visible.
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int64_t* misc = reinterpret_cast<int64_t*>(smem + C::OFF_MISC);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + C::OFF_PLAN);

    // pool bases of the device tier [0] and the host tier [1]: codes K, V,
    // scales K, V, zero-points K, V (read per unit from shared memory rather
    // than held in registers)
    __shared__ const uint8_t* pool_tab[2][6];
    if (threadIdx.x == 0) {
        pool_tab[0][0] = p.c.k_codes;
        pool_tab[0][1] = p.c.v_codes;
        pool_tab[0][2] = static_cast<const uint8_t*>(p.c.k_scales);
        pool_tab[0][3] = static_cast<const uint8_t*>(p.c.v_scales);
        pool_tab[0][4] = static_cast<const uint8_t*>(p.c.k_zeros);
        pool_tab[0][5] = static_cast<const uint8_t*>(p.c.v_zeros);
        pool_tab[1][0] = p.c.hk_codes;
        pool_tab[1][1] = p.c.hv_codes;
        pool_tab[1][2] = static_cast<const uint8_t*>(p.c.hk_scales);
        pool_tab[1][3] = static_cast<const uint8_t*>(p.c.hv_scales);
        pool_tab[1][4] = static_cast<const uint8_t*>(p.c.hk_zeros);
        pool_tab[1][5] = static_cast<const uint8_t*>(p.c.hv_zeros);
    }
    grid_dependency_wait();  // the kernel ahead has completed
    const Plan plan = build_plan<C::THREADS, C::WARPS>(p, prefix, misc);  // contains __syncthreads
    if (blockIdx.x == 0) {
        // publish the plan for the merge kernel: [U, S] then prefix[0..B]
        int64_t* wsplan = reinterpret_cast<int64_t*>(p.ws_l + 2 * (size_t)p.n_ctas * G);
        if (threadIdx.x == 0) {
            wsplan[0] = plan.U;
            wsplan[1] = plan.S;
        }
        int32_t* wp = reinterpret_cast<int32_t*>(wsplan + 2);
        for (int b = threadIdx.x; b <= p.B; b += blockDim.x) wp[b] = prefix[b];
    }
    const int Hkv = p.c.num_kv_heads;
    const int P = p.c.page_size;
    if (p.fuse_merge) {  // empty sequences get zero rows (no CTA's slice touches them)
        for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
            if (prefix[b + 1] != prefix[b]) continue;
            const OutRow row = out_row(p, (int64_t)b * p.Hq * D);
            for (int i = threadIdx.x; i < p.Hq * D; i += blockDim.x) store_out(row, i, 0.0f);
        }
    }
    // The CTA's pieces that span more than one warp's slice, or that continue
    // in another CTA (at most one per warp boundary plus the two ends): listed
    // now, by one thread, from the plan alone, so that the end phase starts
    // with the list ready.  Read after the end phase's barrier.
    EndPiece* eps = reinterpret_cast<EndPiece*>(smem + C::OFF_EPS);
    static_assert(sizeof(EndPiece) <= 48, "room for the list");
    __shared__ int s_np;
    if (threadIdx.x == 0) {
        int np = 0;
        PieceWalk cw;
        cw.begin(plan, prefix, blockIdx.x, plan.S);
        for (; !cw.done(); cw.next()) {
            const Piece pc = cw.get(p);
            const int64_t units = prefix[pc.b + 1] - prefix[pc.b];
            const int64_t a = (int64_t)Hkv * prefix[pc.b] + (int64_t)pc.h * units;
            const int64_t k0 = div_line(a + pc.u_lo, plan.Sw), k1 = div_line(a + pc.u_hi - 1, plan.Sw);
            if (pc.whole && k0 == k1) continue;  // inside one warp's slice: already final
            EndPiece& e = eps[np++];
            e.a = a;
            e.units = units;
            e.k0 = k0;
            e.n = (int)(k1 - k0 + 1);
            e.b = pc.b;
            e.h = pc.h;
            e.slot = pc.whole ? -1 : pc.slot;
        }
        s_np = np;
    }
    uint8_t* ring = smem + C::OFF_STAGES + warp * STAGES_ * C::STAGE;

    // ---------------------------------------------------------------- feed
    // Issues this warp's units, in the order the compute loop below consumes
    // them, STAGES-1 units ahead.  Every call commits exactly one cp.async
    // group (empty once the units run out).
    // Every warp is a worker with its own slice of Sw units of the work line;
    // the CTA's slice is its warps' slices end to end.
    const int64_t worker = (int64_t)blockIdx.x * C::WARPS + warp;
    PieceWalk fw;
    fw.begin(plan, prefix, worker, plan.Sw);
    Piece fpc;
    fpc.b = fpc.h = fpc.u_lo = fpc.u_hi = fpc.len = fpc.slot = 0;
    fpc.whole = false;
    int fu = 0, fua = 0, fub = 0;
    int flp = 0, foff = 0;  // logical page of unit fu and its token offset inside the page
    bool fdone = true;
    int fq = 0;             // pieces the feed has queued for the compute
    bool fnew = false;      // the current piece appends its sequence's new token
    int* PQ = reinterpret_cast<int*>(smem + C::OFF_W + warp * C::W_BYTES + C::W_OFF_PQ);
    auto feed_seek = [&]() {
        fdone = true;
        while (!fw.done()) {
            fpc = fw.get(p);
            fua = fpc.u_lo;
            fub = fpc.u_hi;
            if (fua < fub) {
                fu = fua;
                flp = (fu * UNIT) / P;  // once per piece; then advanced incrementally
                foff = (fu * UNIT) - flp * P;
                fdone = false;
                // the piece holds its sequence's last position: with an append,
                // the new token is quantized at the piece's first unit
                fnew = APP && fpc.len > 0 && (int64_t)fpc.u_hi * UNIT >= fpc.len;
                if (lane == 0) {
                    int* d = PQ + (fq & 7) * 8;
                    d[0] = fpc.b;
                    d[1] = fpc.h;
                    d[2] = fpc.u_lo;
                    d[3] = fpc.u_hi;
                    d[4] = fpc.len;
                    d[5] = fpc.whole ? 1 : 0;
                    d[6] = fpc.slot;
                    d[7] = fnew ? 1 : 0;
                }
                ++fq;
                return;
            }
            fw.next();
        }
        if (lane == 0) PQ[(fq & 7) * 8 + 2] = -1;  // the end of this warp's pieces
    };
    feed_seek();
    int bt_b = -1, bt0 = 0, pid = -1, pid_next = -1;  // block-table batch [bt0, bt0 + 32) and the next one
    uint32_t badmask = 0;                             // stages whose page id was outside the pool
    int ist = 0;                                      // stage the next issue fills
    auto issue_one = [&]() {
        if (!fdone) {
            const int st = ist;
            uint8_t* stg = ring + st * C::STAGE;
            const int lp = flp;  // logical page of this unit
            const int32_t* bt_row = p.block_table + (int64_t)fpc.b * p.max_pages;
            if (fpc.b != bt_b || lp < bt0 || lp >= bt0 + 64) {
                bt_b = fpc.b;
                bt0 = lp;
                pid = (bt0 + lane < p.max_pages) ? __ldg(bt_row + bt0 + lane) : -1;
                pid_next = (bt0 + 32 + lane < p.max_pages) ? __ldg(bt_row + bt0 + 32 + lane) : -1;
            } else if (lp >= bt0 + 32) {
                bt0 += 32;
                pid = pid_next;
                pid_next = (bt0 + 32 + lane < p.max_pages) ? __ldg(bt_row + bt0 + 32 + lane) : -1;
            }
            const int page = __shfl_sync(0xffffffffu, pid, lp - bt0);
            if (fu == fua && fnew) {
                // the new token's bf16 K and V rows of this head and the
                // block-table entry of the sequence's last position, read at the
                // piece's start: brought into L2 now
                constexpr int NP = D * 2 / 16;  // 16-byte pieces of one bf16 row
                const int64_t nr = ((int64_t)fpc.b * Hkv + fpc.h) * D;
                if (lane < 2 * NP)
                    prefetch_l2(reinterpret_cast<const uint8_t*>((lane < NP ? p.k_new : p.v_new) + nr) + 16 * (lane % NP));
                if (lane == 0) prefetch_l2(bt_row + (fpc.len - 1) / P);
            }
            if (fu == fua) {  // the piece's query rows travel with the warp's first unit
                const uint8_t* qsrc =
                    reinterpret_cast<const uint8_t*>(p.q + ((int64_t)fpc.b * p.Hq + (int64_t)fpc.h * G) * D);
                constexpr int NQ = C::Q_BYTES / 16;
#pragma unroll
                for (int k = 0; k < (NQ + 31) / 32; ++k) {
                    const int i = k * 32 + lane;
                    if (NQ % 32 == 0 || i < NQ) cp_async16(stg + C::QO + 16 * i, qsrc + 16 * i);
                }
            }
            if (page >= 0 && page < p.c.num_pages + p.c.host_pages) {
                badmask &= ~(1u << st);
                // the page's tier (warp-uniform): its pool bases from the CTA's table
                const int host = page >= p.c.num_pages;
                const uint8_t* const* tb = pool_tab[host];
                const int64_t row = ((int64_t)(page - (host ? p.c.num_pages : 0)) * Hkv + fpc.h) * P + foff;
                const uint8_t* kc = tb[0] + row * C::CB;
                const uint8_t* vc = tb[1] + row * C::CB;
                constexpr int NC = UNIT * C::CB / 16;  // 16-byte pieces of one code run
#pragma unroll
                for (int k = 0; k < (NC + 31) / 32; ++k) {
                    const int i = k * 32 + lane;
                    if (NC % 32 == 0 || i < NC) {
                        cp_async16(stg + C::KC + 16 * i, kc + 16 * i);
                        cp_async16(stg + C::VC + 16 * i, vc + 16 * i);
                    }
                }
                constexpr int NS = UNIT * C::MB / 16;  // 16-byte pieces of one scale (or zero) run
                const int which = lane / NS, part = lane % NS;
                // lane group `which` copies K scales, V scales, (INT4) K zeros, V zeros
                constexpr int NARR = C::INT4 ? 4 : 2;
                static_assert(C::VS == C::KS + UNIT * C::MB && (!C::INT4 || (C::KZ == C::VS + UNIT * C::MB &&
                                                                               C::VZ == C::KZ + UNIT * C::MB)),
                              "the scale and zero runs are consecutive in the stage");
                if (which < NARR)
                    cp_async16(stg + C::KS + which * (UNIT * C::MB) + 16 * part, tb[2 + which] + row * C::MB + 16 * part);
            } else {
                badmask |= (1u << st);
                if (lane == 0) flag_error(p.err, ERR_BAD_TABLE);
            }
            foff += UNIT;
            if (foff == P) {
                foff = 0;
                ++flp;
            }
            if (++fu == fub) {
                fw.next();
                feed_seek();
            }
        }
        cp_async_commit();
        ist = (ist + 1 == STAGES_) ? 0 : ist + 1;
    };

    // ---------------------------------------------------------------- compute
    const int tid = threadIdx.x;
    uint8_t* wbase = smem + C::OFF_W + warp * C::W_BYTES;
    float* Wt = reinterpret_cast<float*>(wbase);                   // [UNIT][G]
    uint32_t* WB = reinterpret_cast<uint32_t*>(wbase);             // dp4a path: weight words
    float* WQ = reinterpret_cast<float*>(wbase + C::W_OFF_WQ);     // [G]
    float* AL = reinterpret_cast<float*>(wbase + C::W_OFF_AL);     // [G]
    float* ZS = reinterpret_cast<float*>(wbase + C::W_OFF_ZS);     // INT4: [NGR][G]
    // score-lane coordinates
    const int k_tok = lane / C::KL;
    const int k_c0 = (C::SHEAD ? (lane % C::KL) % C::DUP : lane % C::KL) * C::CPL;
    const int k_head = (lane % C::KL) / C::DUP;
    const bool k_writer = (lane % C::DUP) == 0;
    // value-lane coordinates
    const int v_c0 = (lane % C::VL) * C::VCH;
    const int v_tok = lane / C::VL;
    const float qk_scale = p.q_scale;  // softmax scale * log2(e)

#pragma unroll 1
    for (int i = 0; i < STAGES_ - 1; ++i) issue_one();  // prologue
    int cst = 0;  // stage the next computed unit sits in
    __syncwarp();  // the queued pieces are visible to every lane
#pragma unroll 1
    for (int qi = 0;; ++qi) {
        const int* pd = PQ + (qi & 7) * 8;  // this piece (read again at its end)
        const int ua = pd[2];
        if (ua < 0) break;
        const int ub = pd[3];
        const int plen = pd[4];
        const bool pd7 = pd[7] != 0;  // the piece appends its sequence's new token
        if (APP && pd7) {
            // a decode that appends its step's token: before the piece's units
            // (outside the unit loop, so that the quantization shares no
            // registers with the loop's state), the warp quantizes the token by
            // the append's rule (the same device code) into the cache and into
            // its buffer NB, from its bf16 rows (prefetched into L2 by the feed).
            // This warp alone reads that slot in the launch.
            uint8_t* nb = wbase + C::W_OFF_NB;
            constexpr int LPR = D / 16;
            const int r = (lane / LPR) & 1;  // 0: K row, 1: V row (lanes past 2 LPR repeat them)
            const int li = lane % LPR;
            const int64_t nr = ((int64_t)pd[0] * Hkv + pd[1]) * D;
            const uint4* src = reinterpret_cast<const uint4*>((r ? p.v_new : p.k_new) + nr) + li * 2;
            const uint4 raw[2] = {__ldg(src), __ldg(src + 1)};
            const int page = __ldg(p.block_table + (int64_t)pd[0] * p.max_pages + (plen - 1) / P);
            const LaneCodes lc = quantize_lane<SCHEME, LPR>(raw);
            const bool ok = page >= 0 && page < p.c.num_pages + p.c.host_pages;
            if (lane < 2 * LPR) {
                store_lane<SCHEME, D>(lc, nb + r * C::CB, nb + 2 * C::CB + r * C::MB,
                                      nb + 2 * C::CB + (2 + r) * C::MB, 0, li);
                if (ok) {
                    const int tier = page >= p.c.num_pages;
                    const uint8_t* const* tb = pool_tab[tier];
                    const int64_t prow = ((int64_t)(page - (tier ? p.c.num_pages : 0)) * Hkv + pd[1]) * P +
                                         (plen - 1) % P;
                    store_lane<SCHEME, D>(lc, const_cast<uint8_t*>(tb[r]), const_cast<uint8_t*>(tb[2 + r]),
                                          const_cast<uint8_t*>(tb[4 + r]), prow, li);
                }
            }
            if (!ok && lane == 0) flag_error(p.err, ERR_BAD_TABLE);
            __syncwarp();
        }
        uint32_t qw[C::QROWS][C::QW];  // query: INT8/INT4 fixed-point bytes, FP8 fp16 pairs
        float qisum[G];         // INT4: sum of this lane's fixed-point query channels, per head
        float my_sq = 0.0f;     // INT8, INT4: fixed-point step of the lane's score head times the softmax scale
        float m_run = -INFINITY, l_run = 0.0f;
        float o[G][C::VCH];
        float zr[C::GPL];  // INT4: this lane's running sum of p * value zero-point, per group
#pragma unroll
        for (int j = 0; j < C::GPL; ++j) zr[j] = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            qisum[g] = 0.0f;
#pragma unroll
            for (int j = 0; j < C::VCH; ++j) o[g][j] = 0.0f;
        }

        for (int u = ua; u < ub; ++u) {
            issue_one();
            cp_async_wait<STAGES_ - 1>();  // this unit's group has landed
            __syncwarp();
            const int st = cst;
            cst = (cst + 1 == STAGES_) ? 0 : cst + 1;
            const uint8_t* stg = ring + st * C::STAGE;
            if (APP && pd7 && u == ub - 1) {
                // the unit of the sequence's last position: the appended token
                // (quantized at the piece's start into NB) is patched into the
                // staged page, whose copy may predate the cache write
                const uint8_t* nb = wbase + C::W_OFF_NB;
                {
                    uint8_t* sw = ring + st * C::STAGE;
                    const int tl = plen - 1 - u * UNIT;
                    const uint32_t* n32 = reinterpret_cast<const uint32_t*>(nb);
                    for (int i = lane; i < C::CB / 4; i += 32) {
                        reinterpret_cast<uint32_t*>(sw + C::KC + tl * C::CB)[i] = n32[i];
                        reinterpret_cast<uint32_t*>(sw + C::VC + tl * C::CB)[i] = n32[C::CB / 4 + i];
                    }
                    constexpr int MW = C::MB / 4;  // words of one token's scales (or zeros)
                    if (lane < MW) {
                        reinterpret_cast<uint32_t*>(sw + C::KS + tl * C::MB)[lane] = n32[2 * C::CB / 4 + lane];
                        reinterpret_cast<uint32_t*>(sw + C::VS + tl * C::MB)[lane] = n32[2 * C::CB / 4 + MW + lane];
                        if constexpr (C::INT4) {
                            reinterpret_cast<uint32_t*>(sw + C::KZ + tl * C::MB)[lane] = n32[2 * C::CB / 4 + 2 * MW + lane];
                            reinterpret_cast<uint32_t*>(sw + C::VZ + tl * C::MB)[lane] = n32[2 * C::CB / 4 + 3 * MW + lane];
                        }
                    }
                    __syncwarp();
                }
            }
            if (u == ua && C::SHEAD) {
                // ---- this lane's head of the query -> 16-bit fixed point bytes:
                // q ~ sq * qi, qi = 256 hi + lo (hi a signed byte, lo an unsigned
                // byte; error <= sq / 2 per element), sq from the head's max |q|
                const uint16_t* qrow = reinterpret_cast<const uint16_t*>(stg + C::QO) + k_head * D + k_c0;
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < C::CPL; j += 8) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(qrow + j);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w4[i] & 0xFFFFu)),
                                                 fabsf(bf16_bits_to_float(w4[i] >> 16))));
                }
#pragma unroll
                for (int off = C::DUP / 2; off >= 1; off >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                const float inv = amax > 0.0f ? 32767.0f / amax : 0.0f;
                my_sq = (amax / 32767.0f) * qk_scale;
                constexpr int NQW = C::CPL / 4;
#pragma unroll
                for (int j = 0; j < C::CPL; j += 8) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(qrow + j);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
                    int qi[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qi[2 * i] = __float2int_rn(bf16_bits_to_float(w4[i] & 0xFFFFu) * inv);
                        qi[2 * i + 1] = __float2int_rn(bf16_bits_to_float(w4[i] >> 16) * inv);
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int* v = qi + 4 * h2;
                        qw[0][j / 4 + h2] = ((uint32_t)(v[0] >> 8) & 0xFF) | (((uint32_t)(v[1] >> 8) & 0xFF) << 8) |
                                            (((uint32_t)(v[2] >> 8) & 0xFF) << 16) | (((uint32_t)(v[3] >> 8) & 0xFF) << 24);
                        qw[0][NQW + j / 4 + h2] = ((uint32_t)v[0] & 0xFF) | (((uint32_t)v[1] & 0xFF) << 8) |
                                                  (((uint32_t)v[2] & 0xFF) << 16) | (((uint32_t)v[3] & 0xFF) << 24);
                    }
                }
            } else if (u == ua) {
                // ---- query rows of this piece -> fp16 pairs in registers
                const uint16_t* qb = reinterpret_cast<const uint16_t*>(stg + C::QO);
#pragma unroll
                for (int g = 0; g < C::QROWS; ++g) {
                    float qf[C::CPL];
#pragma unroll
                    for (int j = 0; j < C::CPL; j += 8) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(qb + g * D + k_c0 + j);
                        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            qf[j + 2 * i] = bf16_bits_to_float(w4[i] & 0xFFFFu);
                            qf[j + 2 * i + 1] = bf16_bits_to_float(w4[i] >> 16);
                        }
                    }
                    if constexpr (C::INT4) {
                        // 16-bit fixed point per (query head): q ~ sq * qi, qi = 256 hi + lo,
                        // hi a signed byte, lo an unsigned byte (error <= sq / 2 per element)
                        float amax = 0.0f;
#pragma unroll
                        for (int j = 0; j < C::CPL; ++j) amax = fmaxf(amax, fabsf(qf[j]));
#pragma unroll
                        for (int off = C::KL / 2; off >= 1; off >>= 1)
                            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                        const float inv = amax > 0.0f ? 32767.0f / amax : 0.0f;
                        const float sqg = amax / 32767.0f;
                        int qi[C::CPL];
                        int isum = 0;
#pragma unroll
                        for (int j = 0; j < C::CPL; ++j) {
                            qi[j] = __float2int_rn(qf[j] * inv);
                            isum += qi[j];
                        }
                        auto hb = [&](int j) { return (uint32_t)((qi[j] >> 8) & 0xFF); };
                        auto lb = [&](int j) { return (uint32_t)(qi[j] & 0xFF); };
                        {  // per 8-channel word: even-channel and odd-channel bytes
#pragma unroll
                            for (int i = 0; i < C::CPL / 8; ++i) {
                                const int b0 = 8 * i;
                                qw[g][4 * i + 0] = hb(b0) | (hb(b0 + 2) << 8) | (hb(b0 + 4) << 16) | (hb(b0 + 6) << 24);
                                qw[g][4 * i + 1] = hb(b0 + 1) | (hb(b0 + 3) << 8) | (hb(b0 + 5) << 16) | (hb(b0 + 7) << 24);
                                qw[g][4 * i + 2] = lb(b0) | (lb(b0 + 2) << 8) | (lb(b0 + 4) << 16) | (lb(b0 + 6) << 24);
                                qw[g][4 * i + 3] = lb(b0 + 1) | (lb(b0 + 3) << 8) | (lb(b0 + 5) << 16) | (lb(b0 + 7) << 24);
                            }
                            if (g == k_head) my_sq = sqg * qk_scale;
                            qisum[g] = (float)isum;
                        }
                    } else {  // FP8: the query as fp16 pairs of consecutive channels
#pragma unroll
                        for (int i = 0; i < C::QW; ++i) {
                            const __half2 h = __floats2half2_rn(qf[2 * i], qf[2 * i + 1]);
                            qw[g][i] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                    }
                }
            }
            int n_valid = plen - u * UNIT;
            n_valid = n_valid > UNIT ? UNIT : n_valid;
            if (badmask & (1u << st)) n_valid = 0;

            if (n_valid > 0) {
                if constexpr (C::VDP) {
                    if (n_valid < UNIT) {
                        // a partial last unit: past the sequence's end the stage holds
                        // whatever the page does; zeroing those value scales (and
                        // zero-points) makes their weights and zero sums exactly 0
                        // (their p is 0), with no per-token test below
                        uint32_t* vs32 = reinterpret_cast<uint32_t*>(ring + st * C::STAGE + C::VS);
                        uint32_t* vz32 = reinterpret_cast<uint32_t*>(ring + st * C::STAGE + C::VZ);
                        const int i = n_valid * (C::MB / 4) + lane;
                        if (i < UNIT * (C::MB / 4)) {
                            vs32[i] = 0u;
                            if constexpr (C::INT4) vz32[i] = 0u;
                        }
                        __syncwarp();
                    }
                }
                // ---- scores for G heads x UNIT tokens
                float sc[C::PASSES];
#pragma unroll
                for (int pass = 0; pass < C::PASSES; ++pass) {
                    const int t = pass * C::TPP + k_tok;
                    float s;
                    if constexpr (C::INT8) {
                        // this lane's head over its CPL channels of token t, in
                        // NA independent dp4a chains (high and low query bytes)
                        const int8_t* src8 = reinterpret_cast<const int8_t*>(stg + C::KC + t * D + k_c0);
                        constexpr int NQW = C::CPL / 4;
                        constexpr int NA = NQW < 4 ? NQW : 4;
                        int ah[NA], al[NA];
#pragma unroll
                        for (int j = 0; j < NA; ++j) ah[j] = al[j] = 0;
#pragma unroll
                        for (int i = 0; i < NQW; i += NA) {
                            int wv[NA];
                            if constexpr (NA == 4) {
                                const int4 r = *reinterpret_cast<const int4*>(src8 + 4 * i);
                                wv[0] = r.x; wv[1] = r.y; wv[2] = r.z; wv[3] = r.w;
                            } else {
                                const int2 r = *reinterpret_cast<const int2*>(src8 + 4 * i);
                                wv[0] = r.x; wv[1] = r.y;
                            }
#pragma unroll
                            for (int j = 0; j < NA; ++j) {
                                ah[j] = dp4a_ss((int)qw[0][i + j], wv[j], ah[j]);
                                al[j] = dp4a_us(qw[0][NQW + i + j], wv[j], al[j]);
                            }
                        }
                        int hs = 0, ls = 0;
#pragma unroll
                        for (int j = 0; j < NA; ++j) {
                            hs += ah[j];
                            ls += al[j];
                        }
                        int ai = hs * 256 + ls;  // exact: |sum| < 2^30
#pragma unroll
                        for (int off = C::DUP / 2; off >= 1; off >>= 1) ai += __shfl_xor_sync(0xffffffffu, ai, off);
                        s = (float)ai * (my_sq * reinterpret_cast<const float*>(stg + C::KS)[t]);
                    } else if constexpr (C::INT4) {
                        const uint8_t* src = stg + C::KC + t * (D / 2) + k_c0 / 2;
                        uint32_t wv[C::CPL / 8];
                        if constexpr (C::CPL == 16) {
                            const uint2 r = *reinterpret_cast<const uint2*>(src);
                            wv[0] = r.x; wv[1] = r.y;
                        } else {
                            wv[0] = *reinterpret_cast<const uint32_t*>(src);
                        }
                        uint32_t ev[C::CPL / 8], od[C::CPL / 8];
#pragma unroll
                        for (int i = 0; i < C::CPL / 8; ++i) {
                            ev[i] = wv[i] & 0x0F0F0F0Fu;         // even channels as bytes
                            od[i] = (wv[i] >> 4) & 0x0F0F0F0Fu;  // odd channels as bytes
                        }
                        const int gi = t * C::NGR + k_c0 / 32;
                        const float ks = __half2float(reinterpret_cast<const __half*>(stg + C::KS)[gi]);
                        const float kz = __half2float(reinterpret_cast<const __half*>(stg + C::KZ)[gi]);
                        float part[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            int ah = 0, al = 0;
#pragma unroll
                            for (int i = 0; i < C::CPL / 8; ++i) {
                                ah = dp4a_su((int)qw[g][4 * i + 0], ev[i], ah);
                                ah = dp4a_su((int)qw[g][4 * i + 1], od[i], ah);
                                al = dp4a_uu(qw[g][4 * i + 2], ev[i], al);
                                al = dp4a_uu(qw[g][4 * i + 3], od[i], al);
                            }
                            // sum_j qi_j (scale * code_j + zero) over this lane's channels
                            // (one group); the head's step is applied after the reduction
                            part[g] = fmaf(ks, (float)(ah * 256 + al), kz * qisum[g]);
                        }
                        transpose_reduce<float, G, C::KL / 2>(part, lane);
                        s = part[0] * my_sq;
                    } else {
                        constexpr int NA1 = C::TWO_ACC ? G : 1;
                        float acc[G], acc1[NA1];
#pragma unroll
                        for (int g = 0; g < G; ++g) acc[g] = 0.0f;
#pragma unroll
                        for (int g = 0; g < NA1; ++g) acc1[g] = 0.0f;
                        const uint8_t* src = stg + C::KC + t * D + k_c0;
                        uint32_t wv[C::CPL / 4];
                        if constexpr (C::CPL == 16) {
                            const uint4 r = *reinterpret_cast<const uint4*>(src);
                            wv[0] = r.x; wv[1] = r.y; wv[2] = r.z; wv[3] = r.w;
                        } else {
                            const uint2 r = *reinterpret_cast<const uint2*>(src);
                            wv[0] = r.x; wv[1] = r.y;
                        }
#pragma unroll
                        for (int i = 0; i < C::CPL / 4; ++i) {
                            const uint32_t c01 = e4m3x2_to_h2(wv[i]);
                            const uint32_t c23 = e4m3x2_to_h2(wv[i] >> 16);
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                if constexpr (C::TWO_ACC) {
                                    mfma_h2(qw[g][2 * i], c01, acc[g], acc1[g % NA1]);
                                    mfma_h2(qw[g][2 * i + 1], c23, acc[g], acc1[g % NA1]);
                                } else {
                                    mfma_h2_1(qw[g][2 * i], c01, acc[g]);
                                    mfma_h2_1(qw[g][2 * i + 1], c23, acc[g]);
                                }
                            }
                        }
                        if constexpr (C::TWO_ACC) {
#pragma unroll
                            for (int g = 0; g < G; ++g) acc[g] += acc1[g % NA1];
                        }
                        transpose_reduce<float, G, C::KL / 2>(acc, lane);
                        s = acc[0] * (reinterpret_cast<const float*>(stg + C::KS)[t] * qk_scale);
                    }
                    sc[pass] = (t < n_valid) ? s : -INFINITY;
                }
                // ---- online softmax (base 2) on the score lanes
                float mx = sc[0];
#pragma unroll
                for (int pass = 1; pass < C::PASSES; ++pass) mx = fmaxf(mx, sc[pass]);
#pragma unroll
                for (int off = C::KL; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_new = fmaxf(m_run, mx);
                const float alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_new);
                float psum = 0.0f;
                if constexpr (C::VDP) {
                    // weights W = p * value scale (INT4: the scale of each of the
                    // lane's GPL groups), then 16-bit fixed point per (unit, group,
                    // head): W ~ wq * (256 hi + lo), wq = max W / 65535
                    // the weight groups this score lane writes (INT4: GPL groups
                    // from w_r0; INT8: the one group, on the lane that writes its head)
                    const int w_r0 = ((lane % C::DUP) * C::GPL) % C::NGW;
                    const bool w_writer = (lane % C::DUP) * C::GPL < C::NGW;
                    float wv[C::GPL][C::PASSES];
                    float wmax[C::GPL], zs[C::GPL];
#pragma unroll
                    for (int j = 0; j < C::GPL; ++j) wmax[j] = zs[j] = 0.0f;
#pragma unroll
                    for (int pass = 0; pass < C::PASSES; ++pass) {
                        const int t = pass * C::TPP + k_tok;
                        const float pr = fast_exp2(sc[pass] - m_new);  // a masked token (-inf) gives 0
                        psum += pr;
                        if constexpr (C::INT8) {
                            wv[0][pass] = pr * reinterpret_cast<const float*>(stg + C::VS)[t];
                        } else {
                            float vs[C::GPL], vz[C::GPL];
                            load_halves<C::GPL>(stg + C::VS + 2 * (t * C::NGR + w_r0), vs);
                            load_halves<C::GPL>(stg + C::VZ + 2 * (t * C::NGR + w_r0), vz);
#pragma unroll
                            for (int j = 0; j < C::GPL; ++j) {
                                wv[j][pass] = pr * vs[j];
                                zs[j] = fmaf(pr, vz[j], zs[j]);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < C::GPL; ++j) wmax[j] = fmaxf(wmax[j], wv[j][pass]);
                    }
                    // one step per (unit, head) over all its groups: the max of the
                    // head's weights over the token slots and over the lanes that
                    // hold its other groups (or duplicates of them)
                    float wm = wmax[0];
#pragma unroll
                    for (int j = 1; j < C::GPL; ++j) wm = fmaxf(wm, wmax[j]);
#pragma unroll
                    for (int off = C::KL; off < 32; off <<= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
#pragma unroll
                    for (int off = 1; off < C::DUP; off <<= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
                    // Below 1e-30 the unit's weights are negligible next to the
                    // running sum (>= 1 after the first token) and are dropped.
                    const bool live = wm > 1e-30f;
                    const float inv = live ? __fdividef(65535.0f, wm) : 0.0f;
                    if (k_writer && k_tok == 0) WQ[k_head] = live ? wm * (1.0f / 65535.0f) : 0.0f;
#pragma unroll
                    for (int j = 0; j < C::GPL; ++j) {
                        // round to nearest in the low mantissa bits of 2^23 + W * inv;
                        // W * inv <= 65535 (1 + 2^-22) never rounds up to 65536
                        uint32_t bits[C::PASSES];
#pragma unroll
                        for (int pass = 0; pass < C::PASSES; ++pass)
                            bits[pass] = __float_as_uint(fmaf(wv[j][pass], inv, 8388608.0f));
                        // this lane's bytes of its block: low bytes -> lo word, next bytes -> hi word
                        uint32_t lo = __byte_perm(bits[0], bits[1], 0x0040);
                        uint32_t hi = __byte_perm(bits[0], bits[1], 0x0051);
                        if constexpr (C::PASSES == 4) {
                            lo = __byte_perm(lo, __byte_perm(bits[2], bits[3], 0x0040), 0x5410);
                            hi = __byte_perm(hi, __byte_perm(bits[2], bits[3], 0x0051), 0x5410);
                        }
                        if (w_writer) {
                            const int blk = k_tok / C::LPB;
                            const int wi = ((w_r0 + j) * C::NB + blk) * G + k_head;  // hi word; lo is WB_HALF on
                            if constexpr (C::PASSES == 4) {
                                WB[wi] = hi;
                                WB[wi + C::WB_HALF] = lo;
                            } else {
                                uint16_t* wb16 = reinterpret_cast<uint16_t*>(WB);
                                wb16[2 * wi + k_tok % 2] = (uint16_t)hi;
                                wb16[2 * (wi + C::WB_HALF) + k_tok % 2] = (uint16_t)lo;
                            }
                        }
                        if constexpr (C::INT4) zr[j] = fmaf(zr[j], alpha, zs[j]);
                    }
                } else {
#pragma unroll
                    for (int pass = 0; pass < C::PASSES; ++pass) {
                        const int t = pass * C::TPP + k_tok;
                        const float pr = fast_exp2(sc[pass] - m_new);  // a masked token (-inf) gives 0
                        psum += pr;
                        if (k_writer)
                            Wt[t * G + k_head] = (t < n_valid) ? pr * reinterpret_cast<const float*>(stg + C::VS)[t] : 0.0f;
                    }
                }
                l_run = l_run * alpha + psum;
                m_run = m_new;
                if (k_writer && k_tok == 0) AL[k_head] = alpha;
                const bool rescale = __any_sync(0xffffffffu, alpha != 1.0f);
                __syncwarp();
                // ---- values
                if (rescale) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float a = AL[g];
#pragma unroll
                        for (int jj = 0; jj < C::VCH; ++jj) o[g][jj] *= a;
                    }
                }
                if constexpr (C::VDP) {
                    // codes of one 4-token block x this lane's 4 channels,
                    // transposed to one word per channel (token bytes in block
                    // order).  INT4 keeps each odd channel's code in the high
                    // nibble (16 x code), a factor taken out with the step.
                    uint32_t x[C::NBLK][4];
#pragma unroll
                    for (int k = 0; k < C::NBLK; ++k) {
                        const int b = v_tok + k * C::VT;
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int t = (i % C::PASSES) * C::TPP + b * C::LPB + i / C::PASSES;
                            if constexpr (C::INT4)
                                w[i] = *reinterpret_cast<const uint16_t*>(stg + C::VC + t * (D / 2) + v_c0 / 2);
                            else
                                w[i] = *reinterpret_cast<const uint32_t*>(stg + C::VC + t * D + v_c0);
                        }
                        const uint32_t a01 = __byte_perm(w[0], w[1], 0x5140);
                        const uint32_t a23 = __byte_perm(w[2], w[3], 0x5140);
                        if constexpr (C::INT4) {
                            const uint32_t y0 = __byte_perm(a01, a23, 0x5410);  // channels v_c0, v_c0 + 1
                            const uint32_t y1 = __byte_perm(a01, a23, 0x7632);  // channels v_c0 + 2, v_c0 + 3
                            x[k][0] = y0 & 0x0F0F0F0Fu;
                            x[k][1] = y0 & 0xF0F0F0F0u;
                            x[k][2] = y1 & 0x0F0F0F0Fu;
                            x[k][3] = y1 & 0xF0F0F0F0u;
                        } else {
                            const uint32_t b01 = __byte_perm(w[0], w[1], 0x7362);
                            const uint32_t b23 = __byte_perm(w[2], w[3], 0x7362);
                            x[k][0] = __byte_perm(a01, a23, 0x5410);
                            x[k][1] = __byte_perm(a01, a23, 0x7632);
                            x[k][2] = __byte_perm(b01, b23, 0x5410);
                            x[k][3] = __byte_perm(b01, b23, 0x7632);
                        }
                    }
                    // sum over the unit of (256 hi + lo) * code in int32 (INT8:
                    // |sum| < 2^28; INT4: < 16 * 255 * 240 * 257 < 2^28), then one
                    // FMA per accumulator with the step wq
                    const int rv = C::INT4 ? v_c0 / 32 : 0;  // the lane's weight group
                    constexpr int GC = G < 4 ? G : 4;
#pragma unroll
                    for (int g0 = 0; g0 < G; g0 += GC) {
                        int acc[GC][4];
#pragma unroll
                        for (int gg = 0; gg < GC; ++gg)
#pragma unroll
                            for (int j = 0; j < 4; ++j) acc[gg][j] = 0;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            if (half == 1) {
#pragma unroll
                                for (int gg = 0; gg < GC; ++gg)
#pragma unroll
                                    for (int j = 0; j < 4; ++j) acc[gg][j] *= 256;
                            }
#pragma unroll
                            for (int k = 0; k < C::NBLK; ++k) {
                                const int blk = v_tok + k * C::VT;
                                const uint32_t* wsrc = WB + half * C::WB_HALF + (rv * C::NB + blk) * G + g0;
                                uint32_t wq4[GC];
                                if constexpr (GC == 4) {
                                    const uint4 r = *reinterpret_cast<const uint4*>(wsrc);
                                    wq4[0] = r.x; wq4[1] = r.y; wq4[2] = r.z; wq4[3] = r.w;
                                } else if constexpr (GC == 2) {
                                    const uint2 r = *reinterpret_cast<const uint2*>(wsrc);
                                    wq4[0] = r.x; wq4[1] = r.y;
                                } else {
                                    wq4[0] = *wsrc;
                                }
#pragma unroll
                                for (int gg = 0; gg < GC; ++gg)
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        if constexpr (C::INT4) acc[gg][j] = dp4a_uu(wq4[gg], x[k][j], acc[gg][j]);
                                        else acc[gg][j] = dp4a_us(wq4[gg], (int)x[k][j], acc[gg][j]);
                                    }
                            }
                        }
#pragma unroll
                        for (int gg = 0; gg < GC; ++gg) {
                            const float step = WQ[g0 + gg];
                            const float step_odd = C::INT4 ? step * 0.0625f : step;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                o[g0 + gg][j] = fmaf((float)acc[gg][j], (j & 1) ? step_odd : step, o[g0 + gg][j]);
                        }
                    }
                } else {
#pragma unroll(C::V_UNROLL)
                for (int k = 0; k < UNIT / C::VT; ++k) {
                    const int t = v_tok + k * C::VT;
                    if (t < n_valid) {
                        // FP8: this lane's codes of token t, exactly as fp32
                        float c[C::VCH];
                        uint32_t words[C::VCH / 4];
                        if constexpr (C::VCH == 8) {
                            const uint2 r = *reinterpret_cast<const uint2*>(stg + C::VC + t * D + v_c0);
                            words[0] = r.x;
                            words[1] = r.y;
                        } else {
                            words[0] = *reinterpret_cast<const uint32_t*>(stg + C::VC + t * D + v_c0);
                        }
#pragma unroll
                        for (int i = 0; i < C::VCH / 4; ++i) e4m3x4_to_float(words[i], c + 4 * i);
                        float wg[G];
#pragma unroll
                        for (int g = 0; g < G; g += 4) {
                            if constexpr (G >= 4) {
                                const float4 w4 = *reinterpret_cast<const float4*>(Wt + t * G + g);
                                wg[g] = w4.x; wg[g + 1] = w4.y; wg[g + 2] = w4.z; wg[g + 3] = w4.w;
                            } else {
#pragma unroll
                                for (int gg = 0; gg < G; ++gg) wg[gg] = Wt[t * G + gg];
                            }
                        }
#pragma unroll
                        for (int g = 0; g < G; ++g)
#pragma unroll
                            for (int jj = 0; jj < C::VCH; ++jj) o[g][jj] = fmaf(wg[g], c[jj], o[g][jj]);
                    }
                }
                }
            }
            __syncwarp();
        }

        // ---- end of this warp's piece: sum l over the token groups and o over
        // the lanes that share channels; a segment inside this warp's slice
        // is final, any other piece leaves a partial in the warp's slot
#pragma unroll
        for (int off = C::KL; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
        if constexpr (C::INT4) {
            // the zero-point term sum_t p * zero of each (group, head), summed
            // over the token slots, goes to the value lanes through ZS
            const int w_r0 = ((lane % C::DUP) * C::GPL) % C::NGW;
            const bool w_writer = (lane % C::DUP) * C::GPL < C::NGW;
#pragma unroll
            for (int j = 0; j < C::GPL; ++j) {
                float z = zr[j];
#pragma unroll
                for (int off = C::KL; off < 32; off <<= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                if (w_writer && k_tok == 0) ZS[(w_r0 + j) * G + k_head] = z;
            }
            __syncwarp();
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int jj = 0; jj < C::VCH; ++jj) {
                float v = o[g][jj];
#pragma unroll
                for (int off = C::VL; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if constexpr (C::INT4) v += ZS[(v_c0 / 32) * G + g];
                o[g][jj] = v;
            }
        }
        if (pd[5]) {
            const OutRow row = out_row(p, ((int64_t)pd[0] * p.Hq + (int64_t)pd[1] * G) * D);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float lg = __shfl_sync(0xffffffffu, l_run, g * C::DUP);  // lane g*DUP holds head g
                const float inv = (lg > 0.0f) ? 1.0f / lg : 0.0f;
                if (v_tok == 0) {
#pragma unroll
                    for (int jj = 0; jj < C::VCH; jj += 4)
                        store_out4(row, g * D + v_c0 + jj,
                                   make_float4(o[g][jj] * inv, o[g][jj + 1] * inv, o[g][jj + 2] * inv, o[g][jj + 3] * inv));
                }
            }
        } else {
            const int64_t slot = pd[6];
            if (v_tok == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float* dst = p.wp_o + (slot * G + g) * D + v_c0;
#pragma unroll
                    for (int jj = 0; jj < C::VCH; jj += 4)
                        *reinterpret_cast<float4*>(dst + jj) = make_float4(o[g][jj], o[g][jj + 1], o[g][jj + 2], o[g][jj + 3]);
                }
            }
            if (k_writer && k_tok == 0) {
                p.wp_m[slot * G + k_head] = m_run;
                p.wp_l[slot * G + k_head] = l_run;
            }
        }
    }

    // ---- the CTA's pieces that span more than one warp's slice, or that
    // continue in another CTA: combine the partials its warps left, all such
    // pieces at once (at most one per warp boundary plus the two ends)
    cp_async_wait<0>();
    __syncthreads();  // all warps' rows and partials are written; the rings are idle
    const int np = s_np;
    constexpr int NE = G * D / 4;  // float4 elements of one piece's G output rows
    for (int i0 = warp * 32; i0 < np * NE; i0 += C::THREADS) {  // warp-uniform trip count
        const int it = i0 + lane;
        const EndPiece& e = eps[(it < np * NE ? it : i0) / NE];
        const int elem = it % NE;
        merge_element<D, G>(p.wp_o, p.wp_m, p.wp_l, e.a, plan.Sw, e.k0, e.n, elem / (D / 4), (elem % (D / 4)) * 4,
                            lane, it < np * NE,
                            e.slot < 0 ? out_row(p, ((int64_t)e.b * p.Hq + (int64_t)e.h * G) * D) : no_row(),
                            e.slot < 0 ? nullptr : p.ws_o + (int64_t)e.slot * G * D,
                            e.slot < 0 ? nullptr : p.ws_m + (int64_t)e.slot * G,
                            e.slot < 0 ? nullptr : p.ws_l + (int64_t)e.slot * G);
    }
    if (p.fuse_merge) {
        // count this CTA's arrivals on the (at most two) segments it shares
        // with other CTAs, all at once; then merge, element-parallel, those
        // for which it brought the last partial
        __threadfence();
        __syncthreads();  // the CTA's partials are written and visible
        if (tid < np) {
            EndPiece& e = eps[tid];
            if (e.slot >= 0) {
                const unsigned long long n =
                    (unsigned long long)(div_line(e.a + e.units - 1, plan.S) - div_line(e.a, plan.S) + 1);
                if (!count_arrival(p, e.b, e.h, n)) e.slot = -2;  // not the last: nothing to merge
            } else {
                e.slot = -2;  // final rows already written above
            }
        }
        __syncthreads();
        __threadfence();  // see the other CTAs' partials
        for (int i0 = warp * 32; i0 < np * NE; i0 += C::THREADS) {
            const int it = i0 + lane;
            const EndPiece& e = eps[(it < np * NE ? it : i0) / NE];
            const int elem = it % NE;
            const int64_t k0 = div_line(e.a, plan.S), n = div_line(e.a + e.units - 1, plan.S) - k0 + 1;
            merge_element<D, G>(p.ws_o, p.ws_m, p.ws_l, e.a, plan.S, k0, e.slot == -2 ? 0 : (int)n,
                                elem / (D / 4), (elem % (D / 4)) * 4, lane, it < np * NE && e.slot != -2,
                                out_row(p, ((int64_t)e.b * p.Hq + (int64_t)e.h * G) * D), nullptr, nullptr, nullptr);
        }
    }
}


// Shared memory attribute per device, set once (host-only state).  Safe to
// call from several host threads: the attribute call is idempotent, and the
// flag only records that it succeeded.
template <int SCHEME, int D, int G, bool APP>
cudaError_t configure_decode_t() {
    using C = DecodeCfg<SCHEME, D, G>;
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(decode_partial_kernel<SCHEME, D, G, APP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(MAX_SEQS));
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    return cudaSuccess;
}

// Resident CTAs per SM for this instantiation (the persistent grid is this
// times the SM count), taken at the largest shared-memory size any batch
// needs, so that one value serves every call; queried once per device and
// cached (a failed query is not cached).
template <int SCHEME, int D, int G>
int decode_ctas_per_sm_t(int /*B*/) {
    using C = DecodeCfg<SCHEME, D, G>;
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
    if (configure_decode_t<SCHEME, D, G, false>() != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_partial_kernel<SCHEME, D, G, false>, C::THREADS,
                                                      C::smem_bytes(MAX_SEQS)) != cudaSuccess)
        return 0;
    if (n > 0) cached[dev].store(n, std::memory_order_release);
    return n;
}

template <int SCHEME, int D, int G>
cudaError_t launch_decode_partial_t(const DecodeParams& p, cudaStream_t s) {
    using C = DecodeCfg<SCHEME, D, G>;
    const bool app = p.k_new != nullptr;
    cudaError_t e = app ? configure_decode_t<SCHEME, D, G, true>() : configure_decode_t<SCHEME, D, G, false>();
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
    e = app ? cudaLaunchKernelEx(&cfg, decode_partial_kernel<SCHEME, D, G, true>, p)
            : cudaLaunchKernelEx(&cfg, decode_partial_kernel<SCHEME, D, G, false>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int SCHEME>
cudaError_t launch_scheme(const DecodeParams& p, int G_, cudaStream_t s) {
    const int D_ = p.c.head_dim;
    if (D_ == 128) {
        switch (G_) {
            case 1: return launch_decode_partial_t<SCHEME, 128, 1>(p, s);
            case 2: return launch_decode_partial_t<SCHEME, 128, 2>(p, s);
            case 4: return launch_decode_partial_t<SCHEME, 128, 4>(p, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (G_) {
        case 1: return launch_decode_partial_t<SCHEME, 64, 1>(p, s);
        case 2: return launch_decode_partial_t<SCHEME, 64, 2>(p, s);
        case 4: return launch_decode_partial_t<SCHEME, 64, 4>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <int SCHEME>
int ctas_per_sm_scheme(int head_dim, int G_, int B) {
    if (head_dim == 128) {
        switch (G_) {
            case 1: return decode_ctas_per_sm_t<SCHEME, 128, 1>(B);
            case 2: return decode_ctas_per_sm_t<SCHEME, 128, 2>(B);
            case 4: return decode_ctas_per_sm_t<SCHEME, 128, 4>(B);
        }
        return 0;
    }
    switch (G_) {
        case 1: return decode_ctas_per_sm_t<SCHEME, 64, 1>(B);
        case 2: return decode_ctas_per_sm_t<SCHEME, 64, 2>(B);
        case 4: return decode_ctas_per_sm_t<SCHEME, 64, 4>(B);
    }
    return 0;
}

}  // namespace alu
}  // namespace kvq
