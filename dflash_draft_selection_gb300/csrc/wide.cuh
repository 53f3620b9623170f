// wide.cuh -- rows whose sampling filter reaches past their 64 best tokens:
// a draft row with top_k above 64, or with top_p and top_k off.  The filter
// of the pages' sampling (temperature -> top_k -> renormalise -> top_p ->
// renormalise, FreeToken PR 857 "Speed") then keeps a prefix of the row in
// the order key (value descending, lower id first) whose length and mass come
// from a radix select over the ordered value bits, by count (the top_k-th
// token) and by mass (where the cumulative mass reaches top_p), each level a
// pass over the row by the CTA's completion warp with a 256-bin histogram of
// counts and (fp64) masses in shared memory.  Rows whose cut lies within the 64 best
// need no pass.
#pragma once

#include "rowscan.cuh"

namespace dfl {

// Result of the wide filter: the kept prefix has `cut` tokens and mass P,
// relative to the row maximum m (weights 2^((z - m) c) = e^((z - m) / T)).
struct WideCut {
    int64_t cut;
    float P;
    uint64_t key_cut;  // the order key of the last kept token (make_key); 0: every token is kept
};

__device__ __forceinline__ uint32_t wide_key(float x) { return f2ord(x == 0.0f ? 0.0f : x); }

// Histogram (counts, masses) of bits [shift, shift + 8) of the ordered keys of
// the elements of `row` whose key bits above shift + 8 equal `prefix` (all
// elements when shift = 24).  Warp-uniform; the completion warp only.
template <bool BF16>
__device__ void wide_hist(const ScanGeom &g, int64_t row, uint32_t prefix, int shift, float m, float c,
                          ScanSmem::WideHist &h, int lane) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    for (int i = lane; i < 256; i += 32) {
        h.cnt[i] = 0;
        h.mass[i] = 0.0;
    }
    __syncwarp();
    const char *rowp = g.base + row * g.ld_bytes;
    const int64_t nvec = g.V * esz / 16;
    auto take = [&](float x) {
        const uint32_t k = wide_key(x);
        if (shift < 24 && (k >> (shift + 8)) != prefix) return;
        const int bin = static_cast<int>((k >> shift) & 255u);
        atomicAdd(&h.cnt[bin], 1u);
        atomicAdd(&h.mass[bin], static_cast<double>(ex2((x - m) * c)));
    };
#pragma unroll 1
    for (int64_t v0 = lane; v0 < nvec; v0 += 32 * 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t vi = v0 + u * 32;
            v[u] = vi < nvec ? __ldcs(reinterpret_cast<const uint4 *>(rowp) + vi)
                             : make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (v0 + u * 32 >= nvec) continue;
            float x[VE];
            VL::unpack(v[u], x);
#pragma unroll
            for (int e = 0; e < VE; ++e) take(x[e]);
        }
    }
    for (int64_t i = nvec * VE + lane; i < g.V; i += 32) take(VL::scalar(rowp, i));  // the ragged end
    __syncwarp();
}

// Histogram of bits [shift, shift + 8) of ~id for the elements of `row`
// whose ordered value key is vkey and whose ~id bits above shift + 8 equal
// `prefix`: a select over ~id finds ties in increasing id.  Counts only.
template <bool BF16>
__device__ void wide_hist_id(const ScanGeom &g, int64_t row, uint32_t vkey, uint32_t prefix, int shift,
                             ScanSmem::WideHist &h, int lane) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    for (int i = lane; i < 256; i += 32) {
        h.cnt[i] = 0;
        h.mass[i] = 0.0;
    }
    __syncwarp();
    const char *rowp = g.base + row * g.ld_bytes;
    const int64_t nvec = g.V * esz / 16;
    auto take = [&](float x, uint32_t id) {
        if (wide_key(x) != vkey) return;
        const uint32_t k = ~id;
        if (shift < 24 && (k >> (shift + 8)) != prefix) return;
        atomicAdd(&h.cnt[(k >> shift) & 255u], 1u);
    };
#pragma unroll 1
    for (int64_t v0 = lane; v0 < nvec; v0 += 32 * 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t vi = v0 + u * 32;
            v[u] = vi < nvec ? __ldcs(reinterpret_cast<const uint4 *>(rowp) + vi)
                             : make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (v0 + u * 32 >= nvec) continue;
            float x[VE];
            VL::unpack(v[u], x);
#pragma unroll
            for (int e = 0; e < VE; ++e) take(x[e], static_cast<uint32_t>((v0 + u * 32) * VE + e));
        }
    }
    for (int64_t i = nvec * VE + lane; i < g.V; i += 32) take(VL::scalar(rowp, i), static_cast<uint32_t>(i));
    __syncwarp();
}

// The bin where, from the top bin down, the running count (by_mass false)
// or mass reaches `need`; *above_c / *above_m receive the totals of the bins
// above it.  If rounding leaves the mass short of `need`, the lowest bin that
// holds an element.  Warp-uniform.
__device__ __forceinline__ int wide_pick(const ScanSmem::WideHist &h, bool by_mass, double need, int64_t need_c,
                                         int64_t *above_c, double *above_m, int lane) {
    unsigned int c8[8];
    double m8[8];
    unsigned int lc = 0;
    double lm = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int bin = 255 - (lane * 8 + i);
        c8[i] = h.cnt[bin];
        m8[i] = h.mass[bin];
        lc += c8[i];
        lm += m8[i];
    }
    // exclusive scans over the lanes (lane 0 holds the top bins)
    unsigned int bc = lc;
    double bm = lm;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned int tc = __shfl_up_sync(FULL, bc, d);
        const double tm = __shfl_up_sync(FULL, bm, d);
        if (lane >= d) {
            bc += tc;
            bm += tm;
        }
    }
    bc -= lc;
    bm -= lm;
    const bool reach = by_mass ? (bm + lm >= need && lc > 0) : (static_cast<int64_t>(bc) + lc >= need_c);
    uint32_t hit = __ballot_sync(FULL, reach);
    int L;
    if (hit) {
        L = __ffs(hit) - 1;
    } else {
        L = 31 - __clz(__ballot_sync(FULL, lc > 0));  // mass short by rounding: the lowest bin with an element
    }
    int bin = -1;
    unsigned int ac = 0;
    double am = 0.0;
    if (lane == L) {
        ac = bc;
        am = bm;
        int last = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (bin >= 0) continue;
            if (c8[i] > 0) last = i;
            const bool r = by_mass ? (am + m8[i] >= need && c8[i] > 0) : (static_cast<int64_t>(ac) + c8[i] >= need_c);
            if (r) {
                bin = 255 - (lane * 8 + i);
            } else {
                ac += c8[i];
                am += m8[i];
            }
        }
        if (bin < 0) {  // rounding: take the last bin of this lane that holds an element
            bin = 255 - (lane * 8 + (last >= 0 ? last : 7));
            ac = bc;
            am = bm;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (255 - (lane * 8 + i) > bin) {
                    ac += c8[i];
                    am += m8[i];
                }
        }
    }
    bin = __shfl_sync(FULL, bin, L);
    *above_c = __shfl_sync(FULL, ac, L);
    *above_m = __shfl_sync(FULL, am, L);
    return bin;
}

// Radix select over the ordered keys: the key of the token where the count
// (by_mass false: the need_c-th token) or the mass (the first token at which
// the running mass reaches need) is reached, in the order key.  With
// rel_p > 0, need is rel_p times the row's whole mass, summed in fp64 from
// the first level's histogram.  Returns the key; *cnt_above / *mass_above:
// the elements strictly above its value; *ties: how many elements hold its
// value; *need_used: the mass threshold the select used.  Warp-uniform.
template <bool BF16>
__device__ uint32_t wide_select(ScanSmem &sm, const ScanGeom &g, int64_t row, float m, float c, bool by_mass,
                                double need, double rel_p, int64_t need_c, int64_t *cnt_above, double *mass_above,
                                unsigned int *ties, double *need_used, int lane) {
    const int levels = BF16 ? 2 : 4;  // bf16 keys live in the top 16 bits
    uint32_t prefix = 0;
    int64_t ca = 0;
    double ma = 0.0;
    int bin = 0;
    for (int L = 0; L < levels; ++L) {
        const int shift = 24 - 8 * L;
        wide_hist<BF16>(g, row, prefix, shift, m, c, sm.wide, lane);
        if (L == 0 && rel_p > 0.0) {
            double tot = 0.0;
            for (int i = lane; i < 256; i += 32) tot += sm.wide.mass[i];
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) tot += __shfl_xor_sync(FULL, tot, d);
            need = rel_p * tot;
        }
        int64_t ac;
        double am;
        bin = wide_pick(sm.wide, by_mass, need - ma, need_c - ca, &ac, &am, lane);
        ca += ac;
        ma += am;
        prefix = (prefix << 8) | static_cast<uint32_t>(bin);
    }
    *cnt_above = ca;
    *mass_above = ma;
    *need_used = need;
    *ties = sm.wide.cnt[bin];
    __syncwarp();
    return prefix << (32 - 8 * levels);
}

// The id of the n-th (from 1) lowest-id element whose ordered value key is
// vkey: a count select over ~id, four passes.  Warp-uniform.
template <bool BF16>
__device__ uint32_t wide_tie_id(ScanSmem &sm, const ScanGeom &g, int64_t row, uint32_t vkey, int64_t n, int lane) {
    uint32_t prefix = 0;
    int64_t ca = 0;
    for (int L = 0; L < 4; ++L) {
        const int shift = 24 - 8 * L;
        wide_hist_id<BF16>(g, row, vkey, prefix, shift, sm.wide, lane);
        int64_t ac;
        double am;
        const int bin = wide_pick(sm.wide, false, 0.0, n - ca, &ac, &am, lane);
        ca += ac;
        prefix = (prefix << 8) | static_cast<uint32_t>(bin);
    }
    return ~prefix;
}

// The order key of the last kept token when the cut keeps n_t of the ties
// at ordered value key vkey (ties kept lowest id first).
template <bool BF16>
__device__ uint64_t wide_boundary(ScanSmem &sm, const ScanGeom &g, int64_t row, uint32_t vkey, int64_t n_t,
                                  unsigned int ties, int lane) {
    if (n_t >= static_cast<int64_t>(ties)) return static_cast<uint64_t>(vkey) << 32;  // every tie kept
    const uint32_t id = wide_tie_id<BF16>(sm, g, row, vkey, n_t, lane);
    return (static_cast<uint64_t>(vkey) << 32) | static_cast<uint32_t>(~id);
}

// The wide filter's cut for a row with maximum m (raw), total mass S_all
// relative to it, top_k = ek (<= V; > 64) and top_p = tp, given its 64 best
// keys in `list` (R = 2).  Warp-uniform; the completion warp only.
template <bool BF16>
__device__ WideCut wide_cut(ScanSmem &sm, const ScanGeom &g, int64_t row, const WarpList<2> &list, float m,
                            float S_all, float c, int64_t ek, float tp, bool want_key, int lane) {
    WideCut w;
    w.key_cut = 0;
    w.cut = g.V;
    w.P = S_all;
    const bool top_k = ek < g.V;
    if (!top_k && !(tp < 1.0f)) return w;  // no filter: the whole row
    if (!top_k) {
        // top_p alone: does the cut fall within the 64 best?
        float e[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) e[r] = list.k[r] ? ex2((key_val(list.k[r]) - m) * c) : 0.0f;
        const float thr = tp * S_all;
        float base = 0.0f;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float cum = e[r];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float t = __shfl_up_sync(FULL, cum, d);
                if (lane >= d) cum += t;
            }
            cum += base;
            const uint32_t hit = __ballot_sync(FULL, list.k[r] != 0 && cum >= thr);
            if (hit) {
                const int j = __ffs(hit) - 1;
                w.cut = r * 32 + j + 1;
                w.P = __shfl_sync(FULL, cum, j);
                w.key_cut = list.at(static_cast<int>(w.cut) - 1);
                return w;
            }
            base = __shfl_sync(FULL, cum, 31);
        }
    }
    double S_k = S_all;
    uint32_t key_k = 0;
    int64_t n_tk = 0;
    if (top_k) {
        int64_t ca;
        double ma;
        unsigned int ties;
        double unused;
        key_k = wide_select<BF16>(sm, g, row, m, c, false, 0.0, 0.0, ek, &ca, &ma, &ties, &unused, lane);
        n_tk = ek - ca;
        S_k = ma + static_cast<double>(n_tk) * ex2((ord2f(key_k) - m) * c);
        w.cut = ek;
        w.P = static_cast<float>(S_k);
        if (want_key && !(tp < 1.0f)) w.key_cut = wide_boundary<BF16>(sm, g, row, key_k, n_tk, ties, lane);
    }
    if (tp < 1.0f) {
        // top_k off: the threshold is top_p of the whole row's mass, summed in fp64 by the select's
        // first pass (the scan's fp32 sum is coarser than the mass of a token near a deep cut)
        double thr = static_cast<double>(tp) * S_k;
        int64_t ca;
        double ma;
        unsigned int ties;
        const uint32_t key_p = wide_select<BF16>(sm, g, row, m, c, true, thr, top_k ? 0.0 : static_cast<double>(tp), 0,
                                                 &ca, &ma, &ties, &thr, lane);
        if (!top_k || key_p >= key_k) {
            const double wp = ex2((ord2f(key_p) - m) * c);
            int64_t n_tp = wp > 0.0 ? static_cast<int64_t>(ceil((thr - ma) / wp)) : 1;
            if (n_tp < 1) n_tp = 1;
            if (n_tp > static_cast<int64_t>(ties)) n_tp = ties;
            if (top_k && key_p == key_k && n_tp > n_tk) n_tp = n_tk;
            w.cut = ca + n_tp;
            w.P = static_cast<float>(ma + static_cast<double>(n_tp) * wp);
            if (want_key) w.key_cut = wide_boundary<BF16>(sm, g, row, key_p, n_tp, ties, lane);
        } else if (want_key) {
            // rounding put the top_p cut below the top_k-th token: keep the top_k cut
            unsigned int tk_ties = 0;
            int64_t ca2;
            double ma2, unused;
            const uint32_t kk = wide_select<BF16>(sm, g, row, m, c, false, 0.0, 0.0, ek, &ca2, &ma2, &tk_ties, &unused,
                                                  lane);
            w.key_cut = wide_boundary<BF16>(sm, g, row, kk, ek - ca2, tk_ties, lane);
        }
    }
    return w;
}

}  // namespace dfl
