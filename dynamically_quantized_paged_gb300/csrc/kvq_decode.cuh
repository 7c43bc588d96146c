// kvq_decode.cuh -- the pieces of the split-K decode (K2) that do not depend
// on how one slice of work is computed: the split plan, the walk over a
// worker's segment pieces, the log-sum-exp merge of split partials (fused
// into K2's end, or K3, the merge kernel of the two-launch form) and the
// arrival counting that picks the CTA which merges.  The kernel itself is in
// kvq_tc.cuh.
//
// Decomposition.  The work of one call is the sequence of 16-token units of
// every (sequence, KV head) "segment", laid end to end in (b, h, unit) order.
// A persistent grid of n_ctas CTAs (one per SM) cuts that line into equal
// slices of S units, one per CTA.  A segment that lies inside one slice is
// finished by its CTA (final output rows).  A segment cut by slice
// boundaries leaves one partial (running max m, sum l, unnormalized o) per
// CTA it touches, in one of the CTA's two slots (first piece of the slice:
// slot 2k; otherwise 2k + 1); the CTA that delivers the last of them (counted
// in a generation-tagged workspace word) merges them, or, in the two-launch
// form, the merge kernel does.  Slices are a function of logical positions
// only, so physical page placement cannot change the result.
#pragma once

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// ---- final output rows ------------------------------------------------------------
// A final output row (head g's D values at row + g * D): fp32, or bf16 rounded
// to nearest even from the same fp32 value.  base == nullptr: no final row.
struct OutRow {
    void* base;
    int bf16;
};
__device__ __forceinline__ OutRow out_row(const DecodeParams& p, int64_t elem) {
    return OutRow{p.out_bf16 ? static_cast<void*>(static_cast<__nv_bfloat16*>(p.out) + elem)
                             : static_cast<void*>(static_cast<float*>(p.out) + elem),
                  p.out_bf16};
}
__device__ __forceinline__ OutRow no_row() { return OutRow{nullptr, 0}; }
__device__ __forceinline__ void store_out(const OutRow& r, int64_t i, float v) {
    if (r.bf16) static_cast<__nv_bfloat16*>(r.base)[i] = __float2bfloat16_rn(v);
    else static_cast<float*>(r.base)[i] = v;
}
// four consecutive values at i (a multiple of 4)
__device__ __forceinline__ void store_out4(const OutRow& r, int64_t i, float4 v) {
    if (r.bf16) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(r.base) + i) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(r.base) + i) = v;
    }
}

// ---- the split plan ------------------------------------------------------------
// units_b = ceil(min(seq_len_b, max_pages * page_size) / UNIT); segments
// (b, h) laid out in (b, h) order; prefix[b] = sum of units_b' for b' < b;
// U = Hkv * prefix[B]; with WPC workers per CTA, worker slice
// Sw = max(ceil(U / (n_ctas * WPC)), MIN_SLICE_UNITS) and CTA slice
// S = WPC * Sw (the tensor-core kernel: one worker per CTA; the CUDA-core
// kernel: every warp is a worker).
// Quotient of two work-line quantities (unit indices, counts, slice lengths),
// all in [0, 2^32): the host refuses calls whose line has 2^31 units or more,
// so 32-bit division is exact here and much cheaper than 64-bit division.
__device__ __forceinline__ int64_t div_line(int64_t a, int64_t b) { return (int64_t)((uint32_t)a / (uint32_t)b); }

struct Plan {
    int B, Hkv;
    int64_t U;
    int64_t Sw;  // units per worker
    int64_t S;   // units per CTA: its workers' slices laid end to end
};

// All NT threads of the block build the plan: per-sequence unit counts,
// then their exclusive prefix sums in shared memory (prefix[0..B]).
template <int NT, int WPC = 1>
__device__ __forceinline__ Plan build_plan(const DecodeParams& p, int32_t* prefix, int64_t* misc) {
    static_assert(NT % 32 == 0 && NT <= 1024, "whole warps");
    constexpr int NW = NT / 32;
    const int B = p.B;
    const int tid = threadIdx.x;
    const int64_t max_tokens = (int64_t)p.max_pages * p.c.page_size;
    const int chunk = (B + NT - 1) / NT;
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
    __shared__ int tsum[NT];
    tsum[tid] = local;
    __syncthreads();
    if (tid < 32) {
        int v[NW];
        int s = 0;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            v[i] = tsum[tid * NW + i];
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
        for (int i = 0; i < NW; ++i) {
            tsum[tid * NW + i] = run;
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
    const int64_t workers = (int64_t)p.n_ctas * WPC;
    const int64_t Sw = div_line(pl.U + workers - 1, workers);
    pl.Sw = Sw < MIN_SLICE_UNITS ? MIN_SLICE_UNITS : Sw;
    pl.S = pl.Sw * WPC;
    return pl;
}

// One piece of a CTA's slice: the part of one segment that lies in it.
struct Piece {
    int b, h;
    int u_lo, u_hi;   // segment-local units [u_lo, u_hi)
    int len;          // tokens of the sequence (clamped)
    bool whole;       // the piece is the whole segment -> final output
    int slot;         // partial slot otherwise
};

// Walks the segment pieces of CTA k's slice [k S, (k + 1) S).  Holds only
// scalars and the shared-memory prefix pointer (nothing that forces a stack
// frame).
struct PieceWalk {
    const int32_t* prefix;
    int B, Hkv;
    int64_t x, end, worker;
    int b, h, idx;
    __device__ int units(int bb) const { return prefix[bb + 1] - prefix[bb]; }
    __device__ int64_t seg_start(int bb, int hh) const {
        return (int64_t)Hkv * prefix[bb] + (int64_t)hh * units(bb);
    }
    __device__ void begin(const Plan& pl, const int32_t* pre, int64_t k, int64_t S) {
        prefix = pre;
        B = pl.B;
        Hkv = pl.Hkv;
        worker = k;
        x = k * S;
        end = x + S;
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
            h = (int)div_line(x - (int64_t)Hkv * prefix[b], units(b));
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
        pc.slot = (int)(2 * worker + (idx == 0 ? 0 : 1));
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

// Log-sum-exp merge of the partials that workers k0..k1 left for the
// segment starting at work-line unit a.  Workers cut the line in slices of S
// units; worker k's partial of the segment is in slot 2k, or 2k+1 when the
// segment is not the first piece of its slice, of the arrays (so, sm, sl).
// Every thread owns float4 elements of the G x D output rows and merges the
// partials of its head online,
//   M' = max(M, m_k), L' = L 2^(M - M') + l_k 2^(m_k - M'),
//   O' = O 2^(M - M') + o_k 2^(m_k - M'),
// eight partials at a time: each element's o loads are all in flight
// together, and (m_k, l_k) are loaded once per head by one lane each and
// shuffled to the lanes of that head.  The result goes to `row` as O / L
// (final output rows), or, when row is null, to (dst_o, dst_m, dst_l) as a
// partial.  Loads bypass L1: the partials come from other warps and CTAs of
// the same launch.  Every thread of the CTA (NT threads) calls this.
template <int D, int G, int NT>
__device__ __forceinline__ void merge_workers(const float* so, const float* sm, const float* sl, int64_t a,
                                              int64_t S, int64_t k0, int64_t k1, int tid, OutRow row,
                                              float* dst_o, float* dst_m, float* dst_l) {
    constexpr int NE = G * D / 4;                    // float4 elements of the output rows
    constexpr int EPT = (NE + NT - 1) / NT;          // per thread
    constexpr int LPH = D / 4 < 32 ? D / 4 : 32;     // lanes of a warp that share a head
    constexpr int UNR = 8;                           // partials per round
    static_assert(UNR <= LPH, "one lane per partial of a round");
    const int n = (int)(k1 - k0 + 1);
    const int64_t k_start = div_line(a, S);  // the worker whose slice holds the segment's first unit
    const bool start_odd = a != k_start * S;
    const int lane = tid & 31, base = lane / LPH * LPH, sub = lane % LPH;
    auto slot_of = [&](int i) -> int64_t {
        const int64_t k = k0 + i;
        return (k == k_start && start_odd) ? 2 * k + 1 : 2 * k;
    };
    int eg[EPT], ej[EPT];
    float M[EPT], L[EPT];
    float4 O[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
        const int e = tid + k * NT;
        eg[k] = e < NE ? e / (D / 4) : -1;
        ej[k] = (e % (D / 4)) * 4;
        M[k] = -INFINITY;
        L[k] = 0.0f;
        O[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i0 = 0; i0 < n; i0 += UNR) {
        float my_m[EPT], my_l[EPT];
        float4 ov[UNR][EPT];
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            my_m[k] = -INFINITY;
            my_l[k] = 0.0f;
            if (sub < UNR && i0 + sub < n && eg[k] >= 0) {
                const int64_t s = slot_of(i0 + sub);
                my_m[k] = __ldcg(sm + s * G + eg[k]);
                my_l[k] = __ldcg(sl + s * G + eg[k]);
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int64_t s = slot_of(i0 + u);
#pragma unroll
            for (int k = 0; k < EPT; ++k)
                if (i0 + u < n && eg[k] >= 0)
                    ov[u][k] = __ldcg(reinterpret_cast<const float4*>(so + (s * G + eg[k]) * D + ej[k]));
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const float mc = __shfl_sync(0xffffffffu, my_m[k], base + u);
                const float lc = __shfl_sync(0xffffffffu, my_l[k], base + u);
                if (mc == -INFINITY) continue;  // no partial, or one with no tokens
                const float nm = fmaxf(M[k], mc);
                const float fa = (M[k] == -INFINITY) ? 0.0f : fast_exp2(M[k] - nm);
                const float fb = fast_exp2(mc - nm);
                L[k] = fmaf(L[k], fa, lc * fb);
                O[k].x = fmaf(O[k].x, fa, ov[u][k].x * fb);
                O[k].y = fmaf(O[k].y, fa, ov[u][k].y * fb);
                O[k].z = fmaf(O[k].z, fa, ov[u][k].z * fb);
                O[k].w = fmaf(O[k].w, fa, ov[u][k].w * fb);
                M[k] = nm;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
        if (eg[k] < 0) continue;
        if (row.base) {
            const float inv = (L[k] > 0.0f) ? 1.0f / L[k] : 0.0f;
            store_out4(row, eg[k] * D + ej[k], make_float4(O[k].x * inv, O[k].y * inv, O[k].z * inv, O[k].w * inv));
        } else {
            *reinterpret_cast<float4*>(dst_o + eg[k] * D + ej[k]) = O[k];
            if (ej[k] == 0) {
                dst_m[eg[k]] = M[k];
                dst_l[eg[k]] = L[k];
            }
        }
    }
}

// One float4 element (head g, channels j..j+3) of the online log-sum-exp merge
// of the partials workers k0..k0+n-1 left for the segment starting at unit
// a (slices of S units; slot rule as in merge_workers).  Called by all 32
// lanes of a warp together (active = this lane has an element); the lanes
// that share a head share their (m, l) loads by shuffle.  Writes O / L to
// row, or (O, M, L) to the destination partial.
template <int D, int G>
__device__ __forceinline__ void merge_element(const float* so, const float* sm, const float* sl, int64_t a,
                                              int64_t S, int64_t k0, int n, int g, int j, int lane, bool active,
                                              OutRow row, float* dst_o, float* dst_m, float* dst_l) {
    constexpr int LPH = D / 4 < 32 ? D / 4 : 32;
    constexpr int UNR = 8;
    const int64_t k_start = div_line(a, S);
    const bool start_odd = a != k_start * S;
    const int base = lane / LPH * LPH, sub = lane % LPH;
    auto slot_of = [&](int i) -> int64_t {
        const int64_t k = k0 + i;
        return (k == k_start && start_odd) ? 2 * k + 1 : 2 * k;
    };
    // lanes of one head come from the same piece: n is uniform over them
    float M = -INFINITY, L = 0.0f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    const int nmax = __reduce_max_sync(0xffffffffu, active ? n : 0);
    for (int i0 = 0; i0 < nmax; i0 += UNR) {
        float my_m = -INFINITY, my_l = 0.0f;
        if (active && sub < UNR && i0 + sub < n) {
            const int64_t s = slot_of(i0 + sub);
            my_m = __ldcg(sm + s * G + g);
            my_l = __ldcg(sl + s * G + g);
        }
        float4 ov[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u)
            if (active && i0 + u < n)
                ov[u] = __ldcg(reinterpret_cast<const float4*>(so + (slot_of(i0 + u) * G + g) * D + j));
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const float mc = __shfl_sync(0xffffffffu, my_m, base + u);
            const float lc = __shfl_sync(0xffffffffu, my_l, base + u);
            if (!active || i0 + u >= n || mc == -INFINITY) continue;
            const float nm = fmaxf(M, mc);
            const float fa = (M == -INFINITY) ? 0.0f : fast_exp2(M - nm);
            const float fb = fast_exp2(mc - nm);
            L = fmaf(L, fa, lc * fb);
            O.x = fmaf(O.x, fa, ov[u].x * fb);
            O.y = fmaf(O.y, fa, ov[u].y * fb);
            O.z = fmaf(O.z, fa, ov[u].z * fb);
            O.w = fmaf(O.w, fa, ov[u].w * fb);
            M = nm;
        }
    }
    if (!active) return;
    if (row.base) {
        const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
        store_out4(row, g * D + j, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    } else {
        *reinterpret_cast<float4*>(dst_o + g * D + j) = O;
        if (j == 0) {
            dst_m[g] = M;
            dst_l[g] = L;
        }
    }
}

// One-launch form: count one CTA's arrival on segment (b, h), which n CTAs
// touch; returns true for the CTA that brings the last partial (it merges
// them).  The counter holds (generation << 32) | arrivals.  An arrival adds 1
// and reads the old value back in the same atomic; if the old value carries
// this call's generation, the arrival is counted.  Otherwise the word is left
// over from an earlier call (or is garbage), and the CTA installs
// (generation << 32) | 1 with a compare-and-swap, or finds that another CTA
// did and adds again.  Every CTA is counted exactly once.  Only the first
// arrivals of a call can meet a stale word, so the rest take a single atomic
// and contention stays low even when dozens of CTAs arrive together.  No CTA
// waits on another.  The generation is odd, so a cleared word is stale.  One
// thread calls this, after the CTA's partial is written and fenced.  Kept out
// of line: it is off the main loop's path.  Each failed compare-and-swap means
// another arrival changed the word, so the retries are bounded by the
// arrivals; a hard cap on them (flagged as a timeout, nothing merged) guards
// against a word that something outside this call keeps rewriting.  A stale
// word whose low half is all ones turns, with this call's add, into this
// generation with count 0: the next arrival reads it as valid and counts
// itself first, and the arrival whose add made the carry sees a stale value,
// fails its compare-and-swap against the counted word and adds again, so the
// counts stay exact.
static __device__ __noinline__ bool count_arrival(const DecodeParams& p, int b, int h, unsigned long long n) {
    unsigned long long* ctr = p.seg_ctr + (int64_t)b * p.c.num_kv_heads + h;
    const unsigned long long tag = (unsigned long long)p.gen << 32;
    constexpr unsigned long long HI = 0xFFFFFFFF00000000ull, LO = 0xFFFFFFFFull;
    const unsigned long long old = atomicAdd(ctr, 1ull);  // the value before this add
    unsigned long long count;
    if ((old & HI) == tag) {
        count = (old & LO) + 1;
    } else {
        unsigned long long expect = old + 1;  // the word just after this add, if untouched
        for (int tries = 0;; ++tries) {
            if (tries == (1 << 20)) {
                flag_error(p.err, ERR_TIMEOUT);
                return false;
            }
            const unsigned long long seen = atomicCAS(ctr, expect, tag | 1ull);
            if (seen == expect) {  // installed this call's generation, counted as the first
                count = 1;
                break;
            }
            if ((seen & HI) == tag) {  // another arrival installed it: count by adding
                count = (atomicAdd(ctr, 1ull) & LO) + 1;
                break;
            }
            expect = seen;  // other stale adds moved the word: install over it
        }
    }
    // The last arrival clears the word: no other CTA touches it again in this
    // call, and a cleared word reads as stale to the next call, so a replayed
    // call (same generation) starts over too.
    if (count == n) atomicExch(ctr, 0ull);
    return count == n;
}

// ---- K3: merge ------------------------------------------------------------------
// One CTA per (sequence, KV head) segment.  Empty segments get zero rows;
// segments inside one CTA's slice were finished by K2; the others combine the
// partials of CTAs c_first..c_last:  M = max m_c, L = sum l_c 2^(m_c - M),
// out = sum o_c 2^(m_c - M) / L.
template <int D, int G>
__global__ void __launch_bounds__(MERGE_THREADS) decode_merge_kernel(const DecodeParams p) {
    const int b = blockIdx.x / p.c.num_kv_heads;
    const int h = blockIdx.x % p.c.num_kv_heads;
    const int64_t* wsplan = reinterpret_cast<const int64_t*>(p.ws_l + 2 * (size_t)p.n_ctas * G);
    const int64_t S = wsplan[1];
    const int32_t* prefix = reinterpret_cast<const int32_t*>(wsplan + 2);
    const int units = prefix[b + 1] - prefix[b];
    if (units == 0) {
        const OutRow out = out_row(p, ((int64_t)b * p.Hq + (int64_t)h * G) * D);
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) store_out(out, i, 0.0f);
        return;
    }
    const int64_t a = (int64_t)p.c.num_kv_heads * prefix[b] + (int64_t)h * units;
    if (div_line(a, S) == div_line(a + units - 1, S)) return;  // finished inside one CTA's slice
    merge_workers<D, G, MERGE_THREADS>(p.ws_o, p.ws_m, p.ws_l, a, S, div_line(a, S), div_line(a + units - 1, S), threadIdx.x,
                                       out_row(p, ((int64_t)b * p.Hq + (int64_t)h * G) * D), nullptr, nullptr, nullptr);
}

template <int D, int G>
cudaError_t launch_decode_merge_t(const DecodeParams& p, cudaStream_t s) {
    const int64_t n = (int64_t)p.B * p.c.num_kv_heads;
    decode_merge_kernel<D, G><<<(unsigned)n, MERGE_THREADS, 0, s>>>(p);
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

cudaError_t launch_decode_partial_int8(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_partial_fp8(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_partial_int4(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_partial_int4sym(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_partial_int8kc(const DecodeParams& p, int G, cudaStream_t s);
int decode_ctas_per_sm_int8(int head_dim, int G, int B);
int decode_ctas_per_sm_fp8(int head_dim, int G, int B);
int decode_ctas_per_sm_int4(int head_dim, int G, int B);
int decode_ctas_per_sm_int4sym(int head_dim, int G, int B);
int decode_ctas_per_sm_int8kc(int head_dim, int G, int B);

}  // namespace kvq
