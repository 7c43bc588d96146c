// kvq_decode.cuh -- split-K fused-dequantization paged GQA decode attention
// (K2) and the log-sum-exp merge of its splits (K3).
//
// What it computes ("What is KV Cache Optimization? ...", section "Technical
// Architecture", stage "Fused Dequantization Attention Kernel"; "Dynamic KV
// Cache Quantization for Fast LLM Inference", section "Recap of KV Caching"):
// for sequence b and query head g (KV head h = g / G), softmax over every
// cached token t < seq_len of <q, K_t> / sqrt(d), applied to V_t, where K_t and
// V_t are dequantized from their codes inside the kernel and the pages of the
// sequence are found through its block table.
//
// Decomposition (GB300 design).  The work of one call is the sequence of
// 16-token units of every (sequence, KV head) "segment", laid end to end in
// (b, h, unit) order.  A persistent grid of n_ctas CTAs cuts that line into
// equal slices of S units; a CTA walks the segment pieces of its slice.  A
// piece that is a whole segment yields the final output row directly; a
// segment cut by slice boundaries leaves one partial (running max m, sum l,
// unnormalized o) per CTA that touches it, at most two per CTA, and the merge
// kernel combines them.  Slices are a function of logical positions only, so
// physical page placement cannot change the result.
//
// Inside a CTA: warp 4 is the producer.  For every unit it looks up the
// physical page in the block table and issues 1-D bulk copies (TMA) of the K
// codes, V codes and scales (and INT4 zero-points) of those 16 tokens into a
// stage of a per-consumer-warp ring, completing on an mbarrier; the query
// rows of each piece are bulk-copied too.  Warps 0-3 consume units round
// robin:
//  * scores: each lane holds 16 channels of the G query rows as fp16 and
//    turns 16 codes into fp16 with byte permutes (INT8, INT4: exact integer
//    plus a constant bias removed once per score) or the E4M3 converter;
//    mixed-precision FMAs (fp16 x fp16 -> fp32) form partial dots, a
//    transpose-reduction across the lanes sharing a token leaves one score
//    per lane, and the per-token scale is applied once;
//  * online softmax in base 2 directly on those lanes (max over the unit by
//    two shuffles), weights p*scale to shared memory;
//  * values: each lane owns 8 channels x G heads of fp32 accumulators,
//    updated with packed fp32x2 FMAs on exactly converted codes.
// At the end of a piece the four warps' states are combined in shared memory.
#pragma once

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

template <int SCHEME, int D, int G>
struct DecodeCfg {
    static constexpr bool INT4 = SCHEME == KVQ_INT4_ASYM_G32;
    static constexpr bool INT8 = SCHEME == KVQ_INT8_SYM_TOKEN;
    static constexpr int CB = INT4 ? D / 2 : D;        // code bytes per token row
    static constexpr int NGR = D / 32;                 // INT4 groups per row
    static constexpr int MB = INT4 ? NGR * 2 : 4;      // bytes per token in one scale/zero array
    // stage layout (bytes)
    static constexpr int KC = 0;
    static constexpr int VC = KC + UNIT * CB;
    static constexpr int KS = VC + UNIT * CB;
    static constexpr int VS = KS + UNIT * MB;
    static constexpr int KZ = VS + UNIT * MB;
    static constexpr int VZ = KZ + (INT4 ? UNIT * MB : 0);
    static constexpr int STAGE = VZ + (INT4 ? UNIT * MB : 0);
    static constexpr uint32_t STAGE_TX = STAGE;  // bytes one stage receives
    static constexpr int STAGES = STAGE >= 4096 ? 3 : 4;  // ring depth per consumer warp
    // occupancy target: CTAs per SM the register budget is compiled for
    static constexpr int MIN_CTAS = (G >= 8) ? 2 : 3;
    // scores: KL lanes per token, CPL channels per lane, TPP tokens per pass
    static constexpr int CPL = (D == 64 && G == 8) ? 8 : 16;
    static constexpr int KL = D / CPL;
    static constexpr int TPP = 32 / KL;
    static constexpr int PASSES = UNIT / TPP;
    static constexpr int DUP = KL / G;  // lanes that end holding the same (token, head) score
    static constexpr int QW = CPL / 2;  // fp16 pairs of query per head per lane
    static constexpr bool TWO_ACC = G <= 2;  // a second accumulator set for more ILP when registers allow
    // values: VCH channels per lane, VL lanes per token, VT token groups
    static constexpr int VCH = (G >= 8 && D == 128) ? 4 : 8;
    static constexpr int VP = VCH / 2;  // fp32 pairs per head per lane
    static constexpr int VL = D / VCH;
    static constexpr int VT = 32 / VL;
    static constexpr int V_UNROLL = (G >= 8) ? 2 : UNIT / VT;  // token loop unrolling (register pressure)
    // shared memory layout (bytes)
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_Q = OFF_STAGES + CONSUMER_WARPS * STAGES * STAGE;
    static constexpr int Q_BYTES = G * D * 2;
    static constexpr int OFF_CO = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_CM = OFF_CO + CONSUMER_WARPS * G * D * 4;
    static constexpr int OFF_CL = OFF_CM + CONSUMER_WARPS * G * 4;
    static constexpr int OFF_W = (OFF_CL + CONSUMER_WARPS * G * 4 + 15) / 16 * 16;
    // per warp: weight pairs Wt[UNIT][G] (w, w) as 8 bytes, then alpha[G]
    static constexpr int W_BYTES = (UNIT * G * 8 + G * 4 + 15) / 16 * 16;
    static constexpr int OFF_BAR = OFF_W + CONSUMER_WARPS * W_BYTES;
    static constexpr int NBAR = 2 * CONSUMER_WARPS * STAGES + 4;
    static constexpr int OFF_BAD = OFF_BAR + NBAR * 8;  // per stage "page id was invalid" marks
    static constexpr int OFF_MISC = OFF_BAD + CONSUMER_WARPS * STAGES * 4;
    static constexpr int OFF_PLAN = OFF_MISC + 16;
    static size_t smem_bytes(int B) { return OFF_PLAN + (size_t)(B + 1) * 4; }
    static_assert(G <= KL, "each lane must end the reduction holding one head");
    static_assert(STAGE % 16 == 0 && Q_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
    static_assert(OFF_Q % 16 == 0 && OFF_CO % 16 == 0 && OFF_W % 16 == 0, "alignment");
};

// ---- the split plan ------------------------------------------------------------
// units_b = ceil(min(seq_len_b, max_pages * page_size) / UNIT); segments
// (b, h) laid out in (b, h) order; prefix[b] = sum of units_b' for b' < b;
// U = Hkv * prefix[B]; slice S = max(ceil(U / n_ctas), MIN_SLICE_UNITS).
struct Plan {
    int B, Hkv;
    int64_t U, S;
};

// All threads of the block build the plan (prefix sums in shared memory).
__device__ __forceinline__ Plan build_plan(const DecodeParams& p, int32_t* prefix, int64_t* misc) {
    const int B = p.B;
    const int nthr = blockDim.x;
    const int tid = threadIdx.x;
    const int64_t max_tokens = (int64_t)p.max_pages * p.c.page_size;
    const int chunk = (B + nthr - 1) / nthr;
    const int b0 = min(B, tid * chunk), b1 = min(B, b0 + chunk);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        int64_t L = p.seq_lens[b];
        if (L < 0 || L > max_tokens) {
            if (blockIdx.x == 0) flag_error(p.err, ERR_BAD_TABLE);
            L = L < 0 ? 0 : max_tokens;
        }
        const int u = (int)((L + UNIT - 1) / UNIT);
        prefix[b] = u;  // the count, replaced by the exclusive prefix below
        local += u;
    }
    // exclusive scan of the per-thread sums by warp 0
    __shared__ int tsum[DECODE_THREADS];
    tsum[tid] = local;
    __syncthreads();
    if (tid < 32) {
        constexpr int PER = (DECODE_THREADS + 31) / 32;
        int v[PER];
        int s = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int k = tid * PER + i;
            v[i] = (k < nthr) ? tsum[k] : 0;
            s += v[i];
        }
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, off);
            if (tid >= off) incl += n;
        }
        int run = incl - s;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int k = tid * PER + i;
            if (k < nthr) tsum[k] = run;
            run += v[i];
        }
        if (tid == 31) misc[0] = incl;  // total units per head
    }
    __syncthreads();
    int run = tsum[tid];
    for (int b = b0; b < b1; ++b) {  // entries [b0, b1) belong to this thread alone
        const int u = prefix[b];
        prefix[b] = run;
        run += u;
    }
    __syncthreads();
    if (tid == 0) prefix[B] = (int)misc[0];
    __syncthreads();
    Plan pl;
    pl.B = B;
    pl.Hkv = p.c.num_kv_heads;
    pl.U = (int64_t)pl.Hkv * misc[0];
    const int64_t S = (pl.U + p.n_ctas - 1) / p.n_ctas;
    pl.S = S < MIN_SLICE_UNITS ? MIN_SLICE_UNITS : S;
    return pl;
}

// One piece of a CTA's slice.
struct Piece {
    int b, h;
    int u_lo, u_hi;   // segment-local units [u_lo, u_hi)
    int len;          // tokens of the sequence (clamped)
    bool whole;       // the piece is the whole segment -> final output
    int slot;         // partial slot otherwise
};

// Walks the segment pieces of one CTA's slice.  Holds only scalars and the
// shared-memory prefix pointer (nothing that forces a stack frame).
struct PieceWalk {
    const int32_t* prefix;
    int B, Hkv;
    int64_t x, end;
    int b, h, idx, cta;
    __device__ int units(int bb) const { return prefix[bb + 1] - prefix[bb]; }
    __device__ int64_t seg_start(int bb, int hh) const {
        return (int64_t)Hkv * prefix[bb] + (int64_t)hh * units(bb);
    }
    __device__ void begin(const Plan& pl, const int32_t* pre, int c) {
        prefix = pre;
        B = pl.B;
        Hkv = pl.Hkv;
        cta = c;
        x = (int64_t)c * pl.S;
        end = x + pl.S;
        if (end > pl.U) end = pl.U;
        idx = 0;
        b = h = 0;
        if (x < end) {  // segment containing x: smallest b with Hkv*prefix[b+1] > x
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if ((int64_t)Hkv * prefix[mid + 1] > x) hi = mid;
                else lo = mid + 1;
            }
            b = lo;
            h = (int)((x - (int64_t)Hkv * prefix[b]) / units(b));
        }
    }
    __device__ bool done() const { return x >= end; }
    __device__ Piece get(const DecodeParams& p) const {
        Piece pc;
        pc.b = b;
        pc.h = h;
        const int64_t a = seg_start(b, h);
        const int n = units(b);
        const int64_t e = a + n;
        pc.u_lo = (int)(x - a);
        pc.u_hi = (int)((end < e ? end : e) - a);
        const int64_t max_tokens = (int64_t)p.max_pages * p.c.page_size;
        int64_t L = p.seq_lens[b];
        L = L < 0 ? 0 : (L > max_tokens ? max_tokens : L);
        pc.len = (int)L;
        pc.whole = (pc.u_lo == 0 && pc.u_hi == n);
        pc.slot = 2 * cta + (idx == 0 ? 0 : 1);
        return pc;
    }
    __device__ void next() {
        const int64_t e = seg_start(b, h) + units(b);
        x = e < end ? e : end;
        ++idx;
        if (x >= end) return;
        if (++h == Hkv) {
            h = 0;
            do { ++b; } while (units(b) == 0);
        }
    }
};

// Transpose-reduction across the KL lanes that share a token: N values per
// lane in, one (fully summed) value out; the lane ends with head
// (lane % KL) / (KL / G).
template <int N, int OFF>
__device__ __forceinline__ void transpose_reduce(float* v, int lane) {
    if constexpr (OFF >= 1) {
        if constexpr (N > 1) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = upper ? v[i] : v[i + N / 2];
                const float keep = upper ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            transpose_reduce<N / 2, OFF / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            transpose_reduce<1, OFF / 2>(v, lane);
        }
    }
}

template <int SCHEME, int D, int G>
__global__ void __launch_bounds__(DECODE_THREADS, (DecodeCfg<SCHEME, D, G>::MIN_CTAS))
decode_partial_kernel(const DecodeParams p) {
    using C = DecodeCfg<SCHEME, D, G>;
    constexpr int STAGES_ = C::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                                   // [CW][STAGES]
    uint64_t* empty = bars + CONSUMER_WARPS * STAGES_;       // [CW][STAGES]
    uint64_t* qfull = bars + 2 * CONSUMER_WARPS * STAGES_;   // [2]
    uint64_t* qempty = qfull + 2;                            // [2]
    int32_t* bad = reinterpret_cast<int32_t*>(smem + C::OFF_BAD);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    int64_t* misc = reinterpret_cast<int64_t*>(smem + C::OFF_MISC);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + C::OFF_PLAN);

    if (threadIdx.x == 0) {
        for (int i = 0; i < CONSUMER_WARPS * STAGES_; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    const Plan plan = build_plan(p, prefix, misc);  // contains __syncthreads
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

    if (warp == CONSUMER_WARPS) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = l2_evict_first_policy();
        int cnt0 = 0, cnt1 = 0, cnt2 = 0, cnt3 = 0;
        PieceWalk walk;
        walk.begin(plan, prefix, blockIdx.x);
        int pi = 0;
        for (; !walk.done(); walk.next(), ++pi) {
            const Piece pc = walk.get(p);
            if (lane == 0 && !*abort_flag) {
                const int qs = pi & 1;
                if (!mbar_wait(&qempty[qs], ((pi >> 1) & 1) ^ 1)) {
                    flag_error(p.err, ERR_TIMEOUT);
                    *abort_flag = 1;
                } else {
                    mbar_arrive_expect_tx(&qfull[qs], C::Q_BYTES);
                    bulk_load(smem + C::OFF_Q + qs * C::Q_BYTES,
                              p.q + ((int64_t)pc.b * p.Hq + (int64_t)pc.h * G) * D, C::Q_BYTES,
                              &qfull[qs], pol);
                }
            }
            const int32_t* bt_row = p.block_table + (int64_t)pc.b * p.max_pages;
            int batch0 = -1;  // first logical page of the loaded batch
            int pid = -1;
            for (int ub = pc.u_lo; ub < pc.u_hi; ub += CONSUMER_WARPS) {
#pragma unroll
                for (int w = 0; w < CONSUMER_WARPS; ++w) {
                    const int u = ub + w;
                    if (u >= pc.u_hi) break;
                    const int lp = (u * UNIT) / P;  // logical page
                    if (batch0 < 0 || lp >= batch0 + 32) {
                        batch0 = lp;
                        const int k = batch0 + lane;
                        pid = (k < p.max_pages) ? __ldg(bt_row + k) : -1;
                    }
                    const int page = __shfl_sync(0xffffffffu, pid, lp - batch0);
                    int& cnt = (w == 0) ? cnt0 : (w == 1) ? cnt1 : (w == 2) ? cnt2 : cnt3;
                    if (lane == 0 && !*abort_flag) {
                        const int st = cnt % STAGES_;
                        const int k = cnt / STAGES_;
                        const int bi = w * STAGES_ + st;
                        if (!mbar_wait(&empty[bi], (k & 1) ^ 1)) {
                            flag_error(p.err, ERR_TIMEOUT);
                            *abort_flag = 1;
                        } else if (page < 0 || page >= p.c.num_pages) {
                            flag_error(p.err, ERR_BAD_TABLE);
                            bad[bi] = 1;
                            mbar_arrive(&full[bi]);  // completes the phase with no data
                        } else {
                            bad[bi] = 0;
                            const int64_t row = ((int64_t)page * Hkv + pc.h) * P + (u * UNIT) % P;
                            uint8_t* st_ptr = smem + C::OFF_STAGES + bi * C::STAGE;
                            mbar_arrive_expect_tx(&full[bi], C::STAGE_TX);
                            bulk_load(st_ptr + C::KC, p.c.k_codes + row * C::CB, UNIT * C::CB, &full[bi], pol);
                            bulk_load(st_ptr + C::VC, p.c.v_codes + row * C::CB, UNIT * C::CB, &full[bi], pol);
                            bulk_load(st_ptr + C::KS, static_cast<const uint8_t*>(p.c.k_scales) + row * C::MB,
                                      UNIT * C::MB, &full[bi], pol);
                            bulk_load(st_ptr + C::VS, static_cast<const uint8_t*>(p.c.v_scales) + row * C::MB,
                                      UNIT * C::MB, &full[bi], pol);
                            if constexpr (C::INT4) {
                                bulk_load(st_ptr + C::KZ, static_cast<const uint8_t*>(p.c.k_zeros) + row * C::MB,
                                          UNIT * C::MB, &full[bi], pol);
                                bulk_load(st_ptr + C::VZ, static_cast<const uint8_t*>(p.c.v_zeros) + row * C::MB,
                                          UNIT * C::MB, &full[bi], pol);
                            }
                        }
                    }
                    ++cnt;
                }
            }
            __syncwarp();
        }
        // After a timeout, let every copy already issued land before the CTA's
        // shared memory can be reused (bounded again).
        if (lane == 0 && *abort_flag) {
            const int cnts[4] = {cnt0, cnt1, cnt2, cnt3};
            for (int w = 0; w < CONSUMER_WARPS; ++w)
                for (int k = (cnts[w] > STAGES_ ? cnts[w] - STAGES_ : 0); k < cnts[w]; ++k)
                    mbar_wait(&full[w * STAGES_ + k % STAGES_], (k / STAGES_) & 1);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tid = threadIdx.x;  // 0 .. 127
    uint8_t* wbase = smem + C::OFF_W + warp * C::W_BYTES;
    uint64_t* Wt = reinterpret_cast<uint64_t*>(wbase);             // [UNIT][G] (w, w)
    float* AL = reinterpret_cast<float*>(wbase + UNIT * G * 8);    // [G]
    float* CO = reinterpret_cast<float*>(smem + C::OFF_CO);
    float* CM = reinterpret_cast<float*>(smem + C::OFF_CM);
    float* CL = reinterpret_cast<float*>(smem + C::OFF_CL);
    // score-lane coordinates
    const int k_tok = lane / C::KL;
    const int k_c0 = (lane % C::KL) * C::CPL;
    const int k_head = (lane % C::KL) / C::DUP;
    const bool k_writer = (lane % C::DUP) == 0;
    // value-lane coordinates
    const int v_c0 = (lane % C::VL) * C::VCH;
    const int v_tok = lane / C::VL;
    const float qk_scale = p.q_scale;  // softmax scale * log2(e)

    int cnt = 0;
    PieceWalk walk;
    walk.begin(plan, prefix, blockIdx.x);
    int pi = 0;
    for (; !walk.done(); walk.next(), ++pi) {
        const Piece pc = walk.get(p);
        // ---- query rows of this piece -> fp16 pairs in registers
        uint32_t qh[G][C::QW];
        float qsum[G];         // INT4: sum of the query over this lane's channels, per head
        float my_qsum = 0.0f;  // INT8: sum of the query over all channels, this lane's head
        {
            const int qs = pi & 1;
            if (!*abort_flag && !mbar_wait(&qfull[qs], (pi >> 1) & 1)) {
                flag_error(p.err, ERR_TIMEOUT);
                *abort_flag = 1;
            }
            const uint16_t* qb = reinterpret_cast<const uint16_t*>(smem + C::OFF_Q + qs * C::Q_BYTES);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float qf[C::CPL];
#pragma unroll
                for (int j = 0; j < C::CPL; j += 8) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(qb + g * D + k_c0 + j);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qf[j + 2 * i] = __half2float(__float2half_rn(bf16_bits_to_float(w4[i] & 0xFFFFu)));
                        qf[j + 2 * i + 1] = __half2float(__float2half_rn(bf16_bits_to_float(w4[i] >> 16)));
                    }
                }
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < C::CPL; ++j) s += qf[j];
                qsum[g] = s;
#pragma unroll
                for (int i = 0; i < C::QW; ++i) {
                    int a, b2;
                    if constexpr (C::INT4) {  // pair (s, s+4) inside each 8-channel word
                        a = (i / 4) * 8 + (i % 4);
                        b2 = a + 4;
                    } else {                  // consecutive channels
                        a = 2 * i;
                        b2 = 2 * i + 1;
                    }
                    const __half2 h = __floats2half2_rn(qf[a], qf[b2]);
                    qh[g][i] = *reinterpret_cast<const uint32_t*>(&h);
                }
            }
            if constexpr (C::INT8) {  // full-row sums for the bias correction
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int off = C::KL / 2; off >= 1; off >>= 1) qsum[g] += __shfl_xor_sync(0xffffffffu, qsum[g], off);
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (g == k_head) my_qsum = qsum[g];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[qs]);
        }

        float m_run = -INFINITY, l_run = 0.0f;
        uint64_t o[G][C::VP];
        float zacc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            zacc[g] = 0.0f;
#pragma unroll
            for (int j = 0; j < C::VP; ++j) o[g][j] = 0ull;
        }

        for (int j = warp; j < pc.u_hi - pc.u_lo; j += CONSUMER_WARPS, ++cnt) {
            const int st = cnt % STAGES_;
            const int bi = warp * STAGES_ + st;
            bool ok = !*abort_flag;
            if (ok && !mbar_wait(&full[bi], (cnt / STAGES_) & 1)) {
                flag_error(p.err, ERR_TIMEOUT);
                *abort_flag = 1;
                ok = false;
            }
            const int tok0 = (pc.u_lo + j) * UNIT;
            int n_valid = pc.len - tok0;
            n_valid = n_valid > UNIT ? UNIT : n_valid;
            if (!ok || bad[bi]) n_valid = 0;
            const uint8_t* stg = smem + C::OFF_STAGES + bi * C::STAGE;

            if (n_valid > 0) {
                // ---- scores for G heads x UNIT tokens
                float sc[C::PASSES];
#pragma unroll
                for (int pass = 0; pass < C::PASSES; ++pass) {
                    const int t = pass * C::TPP + k_tok;
                    constexpr int NA1 = C::TWO_ACC ? G : 1;
                    float acc[G], acc1[NA1];
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = 0.0f;
#pragma unroll
                    for (int g = 0; g < NA1; ++g) acc1[g] = 0.0f;
                    // acc[g] (+ acc1[g]) += q_g . c over this lane's channels
                    auto dot2 = [&](int g, uint32_t q2, uint32_t c2) {
                        if constexpr (C::TWO_ACC) mfma_h2(q2, c2, acc[g], acc1[g % NA1]);
                        else mfma_h2_1(q2, c2, acc[g]);
                    };
                    if constexpr (!C::INT4) {
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
                            uint32_t c01, c23;
                            if constexpr (C::INT8) {
                                const uint32_t u = wv[i] ^ 0x80808080u;
                                c01 = s8x2_to_h2_biased(u, 0);
                                c23 = s8x2_to_h2_biased(u, 1);
                            } else {
                                c01 = e4m3x2_to_h2(wv[i]);
                                c23 = e4m3x2_to_h2(wv[i] >> 16);
                            }
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                dot2(g, qh[g][2 * i], c01);
                                dot2(g, qh[g][2 * i + 1], c23);
                            }
                        }
                        if constexpr (C::TWO_ACC) {
#pragma unroll
                            for (int g = 0; g < G; ++g) acc[g] += acc1[g % NA1];
                        }
                    } else {
                        const uint8_t* src = stg + C::KC + t * (D / 2) + k_c0 / 2;
                        uint32_t wv[C::CPL / 8];
                        if constexpr (C::CPL == 16) {
                            const uint2 r = *reinterpret_cast<const uint2*>(src);
                            wv[0] = r.x; wv[1] = r.y;
                        } else {
                            wv[0] = *reinterpret_cast<const uint32_t*>(src);
                        }
#pragma unroll
                        for (int i = 0; i < C::CPL / 8; ++i) {
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const uint32_t c2 = u4pair_to_h2_biased(wv[i], s);
#pragma unroll
                                for (int g = 0; g < G; ++g) dot2(g, qh[g][4 * i + s], c2);
                            }
                        }
                        const int gi = t * C::NGR + k_c0 / 32;
                        const float ks = __half2float(reinterpret_cast<const __half*>(stg + C::KS)[gi]);
                        const float kz = __half2float(reinterpret_cast<const __half*>(stg + C::KZ)[gi]);
                        const float zc = fmaf(-U4_H2_BIAS, ks, kz);  // zero - 1024 * scale
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            acc[g] = fmaf(ks, C::TWO_ACC ? acc[g] + acc1[g % NA1] : acc[g], zc * qsum[g]);
                    }
                    transpose_reduce<G, C::KL / 2>(acc, lane);
                    float s;
                    if constexpr (C::INT8) {
                        s = fmaf(-S8_H2_BIAS, my_qsum, acc[0]) * (reinterpret_cast<const float*>(stg + C::KS)[t] * qk_scale);
                    } else if constexpr (C::INT4) {
                        s = acc[0] * qk_scale;
                    } else {
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
#pragma unroll
                for (int pass = 0; pass < C::PASSES; ++pass) {
                    const int t = pass * C::TPP + k_tok;
                    const float pr = (sc[pass] == -INFINITY) ? 0.0f : fast_exp2(sc[pass] - m_new);
                    psum += pr;
                    if (k_writer) {
                        float wv = pr;
                        if constexpr (!C::INT4) wv = (t < n_valid) ? pr * reinterpret_cast<const float*>(stg + C::VS)[t] : 0.0f;
                        Wt[t * G + k_head] = f2pack(wv, wv);
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
                        const uint64_t a2 = f2pack(a, a);
                        zacc[g] *= a;
#pragma unroll
                        for (int jj = 0; jj < C::VP; ++jj) o[g][jj] = fmul2(o[g][jj], a2);
                    }
                }
#pragma unroll(C::V_UNROLL)
                for (int k = 0; k < UNIT / C::VT; ++k) {
                    const int t = v_tok + k * C::VT;
                    if (t < n_valid) {
                        uint64_t c2[C::VP];
                        if constexpr (C::INT8) {
                            const uint64_t bias = f2pack(-8388736.0f, -8388736.0f);
                            uint32_t words[C::VCH / 4];
                            if constexpr (C::VCH == 8) {
                                const uint2 r = *reinterpret_cast<const uint2*>(stg + C::VC + t * D + v_c0);
                                words[0] = r.x;
                                words[1] = r.y;
                            } else {
                                words[0] = *reinterpret_cast<const uint32_t*>(stg + C::VC + t * D + v_c0);
                            }
#pragma unroll
                            for (int i = 0; i < C::VCH / 4; ++i) {
                                const uint32_t u = words[i] ^ 0x80808080u;
                                c2[2 * i] = fadd2(f2pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                                         __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441))), bias);
                                c2[2 * i + 1] = fadd2(f2pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                                             __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443))), bias);
                            }
                        } else if constexpr (!C::INT4) {
                            uint32_t words[C::VCH / 4];
                            if constexpr (C::VCH == 8) {
                                const uint2 r = *reinterpret_cast<const uint2*>(stg + C::VC + t * D + v_c0);
                                words[0] = r.x;
                                words[1] = r.y;
                            } else {
                                words[0] = *reinterpret_cast<const uint32_t*>(stg + C::VC + t * D + v_c0);
                            }
#pragma unroll
                            for (int i = 0; i < C::VP; ++i) {
                                const uint32_t hw = e4m3x2_to_h2(words[i / 2] >> (16 * (i % 2)));
                                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw));
                                c2[i] = f2pack(f.x, f.y);
                            }
                        } else {
                            uint32_t r;
                            if constexpr (C::VCH == 8) r = *reinterpret_cast<const uint32_t*>(stg + C::VC + t * (D / 2) + v_c0 / 2);
                            else r = *reinterpret_cast<const uint16_t*>(stg + C::VC + t * (D / 2) + v_c0 / 2);
                            const uint64_t bias = f2pack(-8388608.0f, -8388608.0f);
#pragma unroll
                            for (int i = 0; i < C::VP; ++i) {
                                const float lo = __uint_as_float(((r >> (8 * i)) & 0xFu) | 0x4B000000u);
                                const float hi = __uint_as_float(((r >> (8 * i + 4)) & 0xFu) | 0x4B000000u);
                                c2[i] = fadd2(f2pack(lo, hi), bias);
                            }
                        }
                        if constexpr (!C::INT4) {
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const uint64_t w2 = Wt[t * G + g];
#pragma unroll
                                for (int jj = 0; jj < C::VP; ++jj) o[g][jj] = ffma2(c2[jj], w2, o[g][jj]);
                            }
                        } else {
                            const int gi = t * C::NGR + v_c0 / 32;
                            const float vs = __half2float(reinterpret_cast<const __half*>(stg + C::VS)[gi]);
                            const float vz = __half2float(reinterpret_cast<const __half*>(stg + C::VZ)[gi]);
                            const uint64_t s2 = f2pack(vs, vs);
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const uint64_t w2 = Wt[t * G + g];
                                float wl, wh;
                                f2unpack(w2, wl, wh);
                                zacc[g] = fmaf(wl, vz, zacc[g]);
                                const uint64_t a2 = fmul2(w2, s2);
#pragma unroll
                                for (int jj = 0; jj < C::VP; ++jj) o[g][jj] = ffma2(c2[jj], a2, o[g][jj]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[bi]);
        }

        // ---- per-warp state -> shared memory
#pragma unroll
        for (int off = C::KL; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int jj = 0; jj < C::VP; ++jj) {
                float lo, hi;
                f2unpack(o[g][jj], lo, hi);
                lo += zacc[g];
                hi += zacc[g];
#pragma unroll
                for (int off = C::VL; off < 32; off <<= 1) {
                    lo += __shfl_xor_sync(0xffffffffu, lo, off);
                    hi += __shfl_xor_sync(0xffffffffu, hi, off);
                }
                o[g][jj] = f2pack(lo, hi);
            }
        }
        if (v_tok == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float f[C::VCH];
#pragma unroll
                for (int jj = 0; jj < C::VP; ++jj) f2unpack(o[g][jj], f[2 * jj], f[2 * jj + 1]);
                float* dst = CO + (warp * G + g) * D + v_c0;
#pragma unroll
                for (int jj = 0; jj < C::VCH; jj += 4)
                    *reinterpret_cast<float4*>(dst + jj) = make_float4(f[jj], f[jj + 1], f[jj + 2], f[jj + 3]);
            }
        }
        if (k_writer && k_tok == 0) {
            CM[warp * G + k_head] = m_run;
            CL[warp * G + k_head] = l_run;
        }
        named_barrier_sync(1, 32 * CONSUMER_WARPS);
        // ---- combine the warps; final row or split partial
        for (int idx = tid; idx < G * D; idx += 32 * CONSUMER_WARPS) {
            const int g = idx / D;
            const int jj = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < CONSUMER_WARPS; ++w) M = fmaxf(M, CM[w * G + g]);
            float L = 0.0f, O = 0.0f;
#pragma unroll
            for (int w = 0; w < CONSUMER_WARPS; ++w) {
                const float mw = CM[w * G + g];
                const float f = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - M);
                L = fmaf(CL[w * G + g], f, L);
                O = fmaf(CO[(w * G + g) * D + jj], f, O);
            }
            if (pc.whole) {
                p.out[((int64_t)pc.b * p.Hq + (int64_t)pc.h * G + g) * D + jj] = (L > 0.0f) ? O / L : 0.0f;
            } else {
                p.ws_o[((int64_t)pc.slot * G + g) * D + jj] = O;
                if (jj == 0) {
                    p.ws_m[pc.slot * G + g] = M;
                    p.ws_l[pc.slot * G + g] = L;
                }
            }
        }
        named_barrier_sync(1, 32 * CONSUMER_WARPS);
    }
}

// ---- K3: merge ------------------------------------------------------------------
// One CTA per (sequence, KV head) segment.  Empty segments get zero rows;
// segments inside one CTA's slice were finished by K2; the others combine the
// partials of CTAs c_first..c_last:  M = max m_c, L = sum l_c 2^(m_c - M),
// out = sum o_c 2^(m_c - M) / L.
template <int D, int G>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
    const int b = blockIdx.x / p.c.num_kv_heads;
    const int h = blockIdx.x % p.c.num_kv_heads;
    const int64_t* wsplan = reinterpret_cast<const int64_t*>(p.ws_l + 2 * (size_t)p.n_ctas * G);
    const int64_t S = wsplan[1];
    const int32_t* prefix = reinterpret_cast<const int32_t*>(wsplan + 2);
    const int units = prefix[b + 1] - prefix[b];
    float* out = p.out + ((int64_t)b * p.Hq + (int64_t)h * G) * D;
    if (units == 0) {
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) out[i] = 0.0f;
        return;
    }
    const int64_t a = (int64_t)p.c.num_kv_heads * prefix[b] + (int64_t)h * units;
    const int64_t e = a + units;
    const int64_t c_first = a / S, c_last = (e - 1) / S;
    if (c_first == c_last) return;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int g = idx / D;
        const int jj = idx % D;
        float M = -INFINITY;
        for (int64_t c = c_first; c <= c_last; ++c) {
            const int64_t slot = (c == c_first && a != c * S) ? 2 * c + 1 : 2 * c;
            M = fmaxf(M, p.ws_m[slot * G + g]);
        }
        float L = 0.0f, O = 0.0f;
        for (int64_t c = c_first; c <= c_last; ++c) {
            const int64_t slot = (c == c_first && a != c * S) ? 2 * c + 1 : 2 * c;
            const float mc = p.ws_m[slot * G + g];
            const float f = (mc == -INFINITY) ? 0.0f : fast_exp2(mc - M);
            L = fmaf(p.ws_l[slot * G + g], f, L);
            O = fmaf(p.ws_o[(slot * G + g) * D + jj], f, O);
        }
        out[g * D + jj] = (L > 0.0f) ? O / L : 0.0f;
    }
}

// Shared memory attribute per device, set once (host-only state).
template <int SCHEME, int D, int G>
cudaError_t configure_decode_t() {
    using C = DecodeCfg<SCHEME, D, G>;
    static int configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(decode_partial_kernel<SCHEME, D, G>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(MAX_SEQS));
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    return cudaSuccess;
}

// Resident CTAs per SM for this instantiation and batch size (the persistent
// grid is this times the SM count).
template <int SCHEME, int D, int G>
int decode_ctas_per_sm_t(int B) {
    using C = DecodeCfg<SCHEME, D, G>;
    if (configure_decode_t<SCHEME, D, G>() != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_partial_kernel<SCHEME, D, G>, DECODE_THREADS,
                                                      C::smem_bytes(B)) != cudaSuccess)
        return 0;
    return n;
}

template <int SCHEME, int D, int G>
cudaError_t launch_decode_partial_t(const DecodeParams& p, cudaStream_t s) {
    using C = DecodeCfg<SCHEME, D, G>;
    cudaError_t e = configure_decode_t<SCHEME, D, G>();
    if (e != cudaSuccess) return e;
    decode_partial_kernel<SCHEME, D, G><<<p.n_ctas, DECODE_THREADS, C::smem_bytes(p.B), s>>>(p);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_decode_merge_t(const DecodeParams& p, cudaStream_t s) {
    const int64_t n = (int64_t)p.B * p.c.num_kv_heads;
    decode_merge_kernel<D, G><<<(unsigned)n, 128, 0, s>>>(p);
    return cudaGetLastError();
}

#define KVQ_DISPATCH_DG(D_, G_, CALL)              \
    do {                                           \
        if ((D_) == 128) {                         \
            switch (G_) {                          \
                case 1: { constexpr int D = 128, G = 1; CALL; } \
                case 2: { constexpr int D = 128, G = 2; CALL; } \
                case 4: { constexpr int D = 128, G = 4; CALL; } \
                default: { constexpr int D = 128, G = 8; CALL; } \
            }                                      \
        }                                          \
        switch (G_) {                              \
            case 1: { constexpr int D = 64, G = 1; CALL; } \
            case 2: { constexpr int D = 64, G = 2; CALL; } \
            case 4: { constexpr int D = 64, G = 4; CALL; } \
            default: { constexpr int D = 64, G = 8; CALL; } \
        }                                          \
    } while (0)

template <int SCHEME>
cudaError_t launch_decode_partial_scheme(const DecodeParams& p, int G_, cudaStream_t s) {
    KVQ_DISPATCH_DG(p.c.head_dim, G_, return (launch_decode_partial_t<SCHEME, D, G>(p, s)));
    return cudaErrorInvalidValue;
}

template <int SCHEME>
int decode_ctas_per_sm_scheme(int head_dim, int G_, int B) {
    KVQ_DISPATCH_DG(head_dim, G_, return (decode_ctas_per_sm_t<SCHEME, D, G>(B)));
    return 0;
}

cudaError_t launch_decode_partial_int8(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_partial_fp8(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_partial_int4(const DecodeParams& p, int G, cudaStream_t s);
int decode_ctas_per_sm_int8(int head_dim, int G, int B);
int decode_ctas_per_sm_fp8(int head_dim, int G, int B);
int decode_ctas_per_sm_int4(int head_dim, int G, int B);

}  // namespace kvq
