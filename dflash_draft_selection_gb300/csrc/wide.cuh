// wide.cuh -- rows whose sampling filter reaches past their 64 best tokens:
// a draft row with top_k above 64, or with top_p and top_k off; a sampled
// target row whose p does the same (or has no filter at all).  The filter of
// the pages' sampling (temperature -> top_k -> renormalise -> top_p ->
// renormalise, FreeToken PR 857 "Speed") then keeps a prefix of the row in
// the order key (value descending, lower id first) whose length and mass come
// from a radix select over the ordered value bits, by count (the top_k-th
// token) and by mass (where the running mass reaches top_p): one pass over
// the row per 8 bits of the value, each a 256-bin histogram of counts and
// masses in shared memory.
//
// The scan kernels finish the rows whose cut their 64 best decide; the
// others the completing CTA marks and, once it has streamed its range,
// finishes in an epilogue on all five of its warps, its stream buffers
// holding the passes' shared memory.
//
// Masses are fixed point: a weight w = 2^((z - m) c) in [0, 1] counts as
// q = round(w 2^s) (s = 40, fewer bits for a vocabulary above 2^23), so that
// sums of up to V of them are exact 64-bit integers whatever the order of
// the additions.  A pass adds each element into its warp's own bins with
// 32-bit shared-memory atomics only (a count, and q as two 20-bit halves),
// and folds the halves into 64-bit register totals every few vectors,
// before a half can overflow.  At the last level a bin is one value, so
// its mass is its count times that value's q and the pass counts only.
#pragma once

#include "rowscan.cuh"

namespace dfl {

constexpr int WIDE_WARPS = SCAN_THREADS / 32;

// The warps that run a pass together, synchronised by the CTA barrier.
struct Team {
    int rank;  // this thread's index in the team
    int size;  // threads
    __device__ __forceinline__ void sync() const { __syncthreads(); }
    __device__ __forceinline__ int warp() const { return rank >> 5; }
};

// Histogram of a pass: counts and 64-bit fixed-point masses (two 32-bit
// halves); a draw's block masses and tie counts reuse it.
struct WideHist {
    union {
        struct {
            unsigned int lo[256], hi[256];
        } fx;
        double blk[256];
    } u;
    unsigned int cnt[256];
};

// Shared memory of the epilogue (in the scan's idle stream buffers).
struct WideSmem {
    WideHist h;
    unsigned int priv[WIDE_WARPS][768];  // each warp's own bins during a pass: counts, q_lo, q_hi
    alignas(16) unsigned char scratch[1024];  // verify's draws
};
static_assert(sizeof(WideSmem) <= sizeof(ScanSmem::buf), "the epilogue's shared memory fits the stream buffers");

__device__ __forceinline__ WideSmem &wide_smem(ScanSmem &sm) { return *reinterpret_cast<WideSmem *>(sm.buf); }

// The wide filter of a row: `cut` tokens of mass P (relative to the row
// maximum) are kept: every token whose value key is above vk, and the nkeep
// lowest ids of the `ties` tokens at value key vk.  all: every token kept.
struct WideCut {
    int64_t cut;
    float P;
    bool all;
    uint32_t vk;
    int64_t nkeep;
    int64_t ties;  // INT64_MAX when not known
};

// Value keys: the order-preserving bits of the logit (-0 as +0); for bf16
// logits the top 16 (the other 16 are the same for every bf16 of a sign).
template <bool BF16>
__device__ __forceinline__ uint32_t wide_vk(float x) {
    const uint32_t k = f2ord(x == 0.0f ? 0.0f : x);
    return BF16 ? k >> 16 : k;
}
template <bool BF16>
__device__ __forceinline__ float wide_vval(uint32_t vk) {
    if (!BF16) return ord2f(vk);
    // a bf16's ordered bits end in 16 zeros (positive) or 16 ones (negative)
    return ord2f((vk << 16) | ((vk & 0x8000u) ? 0u : 0xffffu));
}

// Fixed point: s is the largest value <= 40 with V 2^s < 2^63; q = round(w
// 2^s) = hi 2^20 + lo with hi = floor(w 2^(s - 20)) and lo in [0, 2^20].
struct Fx {
    float shi;   // 2^(s - 20)
    double inv;  // 2^-s
};
__device__ __forceinline__ Fx wide_fx(int64_t V) {
    const int bits = 64 - __clzll(static_cast<unsigned long long>(V));
    const int s = 63 - bits < 40 ? 63 - bits : 40;
    Fx f;
    f.shi = __int_as_float((127 + s - 20) << 23);
    f.inv = __longlong_as_double(static_cast<long long>(1023 - s) << 52);
    return f;
}
__device__ __forceinline__ void wide_q2(float w, const Fx &fx, uint32_t &hi, uint32_t &lo) {
    const float wf = w * fx.shi;  // exact: a power of two
    const float fl = floorf(wf);
    hi = static_cast<uint32_t>(fl);
    lo = static_cast<uint32_t>(rintf((wf - fl) * 1048576.0f));  // wf - fl is exact
}
__device__ __forceinline__ uint64_t wide_q(float w, const Fx &fx) {
    uint32_t hi, lo;
    wide_q2(w, fx, hi, lo);
    return (static_cast<uint64_t>(hi) << 20) + lo;
}

// Sum over the lanes of `grp` of values below 2^45 (exact).
__device__ __forceinline__ uint64_t group_sum_q(unsigned int grp, uint64_t v) {
    const uint32_t l = __reduce_add_sync(grp, static_cast<uint32_t>(v & 0xfffffu));
    const uint32_t h = __reduce_add_sync(grp, static_cast<uint32_t>(v >> 20));
    return (static_cast<uint64_t>(h) << 20) + l;
}
__device__ __forceinline__ void fx_add(unsigned int *lo, unsigned int *hi, uint64_t v) {
    const uint32_t a = static_cast<uint32_t>(v), b = static_cast<uint32_t>(v >> 32);
    const uint32_t old = atomicAdd(lo, a);
    const uint32_t carry = old + a < old ? 1u : 0u;
    if (b + carry) atomicAdd(hi, b + carry);
}
__device__ __forceinline__ uint64_t fx_get(const WideHist &h, int i) {
    return (static_cast<uint64_t>(h.u.fx.hi[i]) << 32) | h.u.fx.lo[i];
}
__device__ __forceinline__ uint64_t shfl_up_u64(uint64_t v, int d) {
    const uint32_t l = __shfl_up_sync(FULL, static_cast<uint32_t>(v), d);
    const uint32_t h = __shfl_up_sync(FULL, static_cast<uint32_t>(v >> 32), d);
    return (static_cast<uint64_t>(h) << 32) | l;
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
    const uint32_t l = __shfl_sync(FULL, static_cast<uint32_t>(v), src);
    const uint32_t h = __shfl_sync(FULL, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(h) << 32) | l;
}

// Calls f(x, valid) for every element of `row`, the team's warps taking
// 32 vectors of 16 bytes in turn, four per lane in flight while the four
// before them are processed; every `fold_every` rounds of four, and at the
// end, fold() (whole warps; lanes past the row see valid false).
template <bool BF16, typename F, typename G>
__device__ __forceinline__ void team_for_each(const Team &tm, const ScanGeom &g, int64_t row, int lane, int fold_every,
                                              F &&f, G &&fold) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    const char *rowp = g.base + row * g.ld_bytes;
    const int64_t nvec = g.V * esz / 16;
    const int64_t step = 4 * static_cast<int64_t>(tm.size);
    auto load = [&](uint4 (&v)[4], int64_t v0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t vi = v0 + u * tm.size + lane;
            v[u] = vi < nvec ? __ldcs(reinterpret_cast<const uint4 *>(rowp) + vi)
                             : make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
        }
    };
    uint4 cur[4], nxt[4];
    int64_t v0 = tm.warp() * 32;
    if (v0 < nvec) load(cur, v0);
    int round = 0;
#pragma unroll 1
    for (; v0 < nvec; v0 += step) {
        if (v0 + step < nvec) load(nxt, v0 + step);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool valid = v0 + u * tm.size + lane < nvec;
            float x[VE];
            VL::unpack(cur[u], x);
#pragma unroll
            for (int e = 0; e < VE; ++e) f(x[e], valid);
        }
        if (++round == fold_every) {
            fold();
            round = 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
    }
    if (tm.warp() == 0) {  // the ragged end (less than one vector)
        for (int64_t i0 = nvec * VE; i0 < g.V; i0 += 32) {
            const int64_t i = i0 + lane;
            f(i < g.V ? VL::scalar(rowp, i) : NEG_INF, i < g.V);
        }
    }
    fold();
}

enum WideMass : int { WM_NONE = 0, WM_ADD = 1, WM_VALUE = 2 };

// Histogram of bits [shift, shift + 8) of the value keys of the elements of
// `row` whose key bits above shift + 8 equal `prefix` (every element at the
// top level) into sm.h: counts, and with WM_ADD the fixed-point masses
// added element by element, with WM_VALUE (the last level, where a bin is
// one value) the count times the value's q.  Team-wide; ends synchronised.
template <bool BF16>
__device__ __forceinline__ void wide_hist(const Team &tm, WideSmem &sm, const ScanGeom &g, int64_t row, uint32_t prefix, int shift,
                          int mass, float m, float c, const Fx &fx, int lane) {
    constexpr int kbits = BF16 ? 16 : 32;
    WideHist &h = sm.h;
    unsigned int *pc = sm.priv[tm.warp()], *pl = pc + 256, *ph = pc + 512;  // the warp's own bins
    for (int i = lane; i < 256; i += 32) {
        pc[i] = 0;
        pl[i] = 0;
        ph[i] = 0;
    }
    for (int i = tm.rank; i < 256; i += tm.size) {
        h.cnt[i] = 0;
        h.u.fx.lo[i] = 0;
        h.u.fx.hi[i] = 0;
    }
    tm.sync();
    const bool top = shift + 8 >= kbits;
    uint64_t tot[8];  // masses of bins lane + 32 j folded so far
#pragma unroll
    for (int j = 0; j < 8; ++j) tot[j] = 0;
    auto fold = [&]() {
        if (mass != WM_ADD) return;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int b = lane + 32 * j;
            tot[j] += (static_cast<uint64_t>(ph[b]) << 20) + pl[b];
            pl[b] = 0;
            ph[b] = 0;
        }
        __syncwarp();
    };
    // a round of four vectors adds at most 4 * 32 * 8 elements of q_hi, q_lo
    // <= 2^20 to a bin: two rounds stay below 2^31
    team_for_each<BF16>(tm, g, row, lane, 2, [&](float x, bool valid) {
        const uint32_t k = wide_vk<BF16>(x);
        if (!valid || (!top && (k >> (shift + 8)) != prefix)) return;
        const int bin = static_cast<int>((k >> shift) & 255u);
        atomicAdd(&pc[bin], 1u);
        if (mass == WM_ADD) {
            uint32_t hi, lo;
            wide_q2(ex2((x - m) * c), fx, hi, lo);
            if (lo) atomicAdd(&pl[bin], lo);
            if (hi) atomicAdd(&ph[bin], hi);
        }
    }, fold);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int b = lane + 32 * j;
        if (pc[b]) atomicAdd(&h.cnt[b], pc[b]);
        if (mass == WM_ADD && tot[j]) fx_add(&h.u.fx.lo[b], &h.u.fx.hi[b], tot[j]);
    }
    tm.sync();
    if (mass == WM_VALUE) {
        if (tm.warp() == 0)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int b = lane + 32 * j;
                const uint32_t vk = (prefix << 8) | static_cast<uint32_t>(b);
                const uint64_t q = static_cast<uint64_t>(h.cnt[b]) * wide_q(ex2((wide_vval<BF16>(vk) - m) * c), fx);
                h.u.fx.lo[b] = static_cast<uint32_t>(q);
                h.u.fx.hi[b] = static_cast<uint32_t>(q >> 32);
            }
        tm.sync();
    }
}

// The bin where, from the top bin down, the running count (by_mass false:
// reaching need_c) or mass (qbase + the bins so far reaching need, in units
// of 2^-s) is reached; *above_c / *above_q: the totals of the bins above it.
// With rel_p > 0, need is first set to rel_p times qbase + the histogram's
// whole mass (*need_io).  If the mass stays short of need, the lowest bin
// that holds an element.  Per warp, from shared memory.
__device__ __forceinline__ int wide_pick(const WideHist &h, bool by_mass, double *need_io, double rel_p,
                                         int64_t need_c, uint64_t qbase, double inv, int64_t *above_c,
                                         uint64_t *above_q, int lane) {
    unsigned int c8[8];
    uint64_t q8[8];
    unsigned int lc = 0;
    uint64_t lq = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int bin = 255 - (lane * 8 + i);
        c8[i] = h.cnt[bin];
        q8[i] = fx_get(h, bin);
        lc += c8[i];
        lq += q8[i];
    }
    // inclusive scans over the lanes (lane 0 holds the top bins)
    unsigned int bc = lc;
    uint64_t bq = lq;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned int tc = __shfl_up_sync(FULL, bc, d);
        const uint64_t tq = shfl_up_u64(bq, d);
        if (lane >= d) {
            bc += tc;
            bq += tq;
        }
    }
    if (rel_p > 0.0) *need_io = rel_p * (static_cast<double>(qbase + shfl_u64(bq, 31)) * inv);
    const double need = *need_io;
    bc -= lc;
    bq -= lq;
    const bool reach = by_mass ? (static_cast<double>(qbase + bq + lq) * inv >= need && lc > 0)
                               : (static_cast<int64_t>(bc) + lc >= need_c);
    const uint32_t hit = __ballot_sync(FULL, reach);
    const int L = hit ? __ffs(hit) - 1 : 31 - __clz(__ballot_sync(FULL, lc > 0));
    int bin = -1;
    unsigned int ac = 0;
    uint64_t aq = 0;
    if (lane == L) {
        ac = bc;
        aq = bq;
        int last = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (bin >= 0) continue;
            if (c8[i] > 0) last = i;
            const bool r = by_mass ? (static_cast<double>(qbase + aq + q8[i]) * inv >= need && c8[i] > 0)
                                   : (static_cast<int64_t>(ac) + c8[i] >= need_c);
            if (r) {
                bin = 255 - (lane * 8 + i);
            } else {
                ac += c8[i];
                aq += q8[i];
            }
        }
        if (bin < 0) {  // short: the last bin of this lane that holds an element
            bin = 255 - (lane * 8 + (last >= 0 ? last : 7));
            ac = bc;
            aq = bq;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (255 - (lane * 8 + i) > bin) {
                    ac += c8[i];
                    aq += q8[i];
                }
        }
    }
    bin = __shfl_sync(FULL, bin, L);
    *above_c = __shfl_sync(FULL, ac, L);
    *above_q = shfl_u64(aq, L);
    return bin;
}

// Radix select over the value keys: the key where the count (by_mass false:
// the need_c-th token) or the mass (the first token at which the running
// mass reaches need; with rel_p > 0, need = rel_p times the row's whole mass,
// summed exactly by the first pass) is reached.  *cnt_above / *q_above: the
// elements strictly above its value; *ties: how many hold it; *need_io: the
// threshold used.  Team-wide.
template <bool BF16>
__device__ uint32_t wide_select(const Team &tm, WideSmem &sm, const ScanGeom &g, int64_t row, float m, float c,
                                const Fx &fx, bool by_mass, double *need_io, double rel_p, int64_t need_c,
                                int64_t *cnt_above, uint64_t *q_above, int64_t *ties, int lane) {
    constexpr int kbits = BF16 ? 16 : 32;
    uint32_t prefix = 0;
    int64_t ca = 0;
    uint64_t qa = 0;
    for (int shift = kbits - 8; shift >= 0; shift -= 8) {
        // a count select still sums the mass above its bin: P is the kept mass
        const int mass = shift == 0 ? WM_VALUE : WM_ADD;
        wide_hist<BF16>(tm, sm, g, row, prefix, shift, mass, m, c, fx, lane);
        int64_t ac;
        uint64_t aq;
        const int bin = wide_pick(sm.h, by_mass, need_io, shift == kbits - 8 ? rel_p : 0.0, need_c - ca, qa,
                                  fx.inv, &ac, &aq, lane);
        if (shift == 0) *ties = sm.h.cnt[bin];
        tm.sync();  // every warp read the histogram before the next pass clears it
        ca += ac;
        qa += aq;
        prefix = (prefix << 8) | static_cast<uint32_t>(bin);
    }
    *cnt_above = ca;
    *q_above = qa;
    return prefix;
}

// The cut when the 64 best keys of the row (`list`, R = 2) decide it: no
// filter, or top_p alone with its cut within them (threshold top_p times
// the scan's total S_all).  Returns false when passes are needed.  Warp.
template <bool BF16>
__device__ bool wide_cut_list(const WarpList<2> &list, float m, float S_all, float c, int64_t ek, float tp,
                              int64_t V, WideCut *out, int lane) {
    WideCut w;
    w.cut = V;
    w.P = S_all;
    w.all = true;
    w.vk = 0;
    w.nkeep = 0;
    w.ties = INT64_MAX;
    *out = w;
    if (ek < V) return false;
    if (!(tp < 1.0f)) return true;  // no filter: the whole row
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
            w.all = false;
            w.vk = wide_vk<BF16>(key_val(list.at(static_cast<int>(w.cut) - 1)));
            // the list holds the lowest ids of a value first: the kept ties are
            // the list's entries of value vk before the cut
            int64_t nk = 0, nt = 0;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const bool same = list.k[rr] != 0 && wide_vk<BF16>(key_val(list.k[rr])) == w.vk;
                nk += __popc(__ballot_sync(FULL, same && rr * 32 + lane < w.cut));
                nt += __popc(__ballot_sync(FULL, same));
            }
            w.nkeep = nk;
            // ties past the list's end are not known
            const uint64_t last = list.at(DFLASH2_MAX_TOPK - 1);
            w.ties = last != 0 && wide_vk<BF16>(key_val(last)) == w.vk ? INT64_MAX : nt;
            *out = w;
            return true;
        }
        base = __shfl_sync(FULL, cum, 31);
    }
    return false;
}

// The cut by passes over the row for top_k = ek (<= V) and top_p = tp, the
// row's maximum m (raw) and c = log2(e) / T.  Team-wide.
template <bool BF16>
__device__ __forceinline__ WideCut wide_cut_passes(const Team &tm, WideSmem &sm, const ScanGeom &g, int64_t row, float m, float c,
                                   int64_t ek, float tp, int lane) {
    const Fx fx = wide_fx(g.V);
    const double inv = fx.inv;
    WideCut w;
    w.cut = g.V;
    w.P = NAN;
    w.all = true;
    w.vk = 0;
    w.nkeep = 0;
    w.ties = INT64_MAX;
    const bool top_k = ek < g.V;
    uint64_t Sq = 0;
    uint32_t vk_k = 0;
    int64_t n_tk = 0;
    if (top_k) {
        int64_t ca, ties;
        uint64_t qa;
        double unused = 0.0;
        vk_k = wide_select<BF16>(tm, sm, g, row, m, c, fx, false, &unused, 0.0, ek, &ca, &qa, &ties, lane);
        n_tk = ek - ca;
        const uint64_t qk = wide_q(ex2((wide_vval<BF16>(vk_k) - m) * c), fx);
        Sq = qa + static_cast<uint64_t>(n_tk) * qk;
        w.cut = ek;
        w.P = static_cast<float>(static_cast<double>(Sq) * inv);
        w.all = false;
        w.vk = vk_k;
        w.nkeep = n_tk;
        w.ties = ties;
    }
    if (tp < 1.0f) {
        // the threshold: top_p of the mass the top_k cut kept, or of the whole
        // row summed exactly by the select's first pass
        double thr = top_k ? static_cast<double>(tp) * (static_cast<double>(Sq) * inv) : 0.0;
        int64_t ca, ties;
        uint64_t qa;
        const uint32_t vk_p = wide_select<BF16>(tm, sm, g, row, m, c, fx, true, &thr,
                                                top_k ? 0.0 : static_cast<double>(tp), 0, &ca, &qa, &ties, lane);
        if (!top_k || vk_p >= vk_k) {
            const uint64_t qp = wide_q(ex2((wide_vval<BF16>(vk_p) - m) * c), fx);
            const double wp = static_cast<double>(qp) * inv;
            int64_t n_tp = wp > 0.0 ? static_cast<int64_t>(ceil((thr - static_cast<double>(qa) * inv) / wp)) : 1;
            if (n_tp < 1) n_tp = 1;
            if (n_tp > ties) n_tp = ties;
            if (top_k && vk_p == vk_k && n_tp > n_tk) n_tp = n_tk;
            w.cut = ca + n_tp;
            w.P = static_cast<float>(static_cast<double>(qa + static_cast<uint64_t>(n_tp) * qp) * inv);
            w.all = false;
            w.vk = vk_p;
            w.nkeep = n_tp;
            w.ties = ties;
        }  // else rounding put the top_p cut below the top_k-th token: the top_k cut stands
    }
    return w;
}

// Where token z of the row stands against the cut: 1 above it (kept), 0
// below, 2 a tie at the cut's value (kept if its rank among the ties, by id,
// is below nkeep).
template <bool BF16>
__device__ __forceinline__ int wide_side(const WideCut &wc, float z) {
    if (wc.all) return 1;
    const uint32_t k = wide_vk<BF16>(z);
    return k > wc.vk ? 1 : (k == wc.vk ? (wc.nkeep >= wc.ties ? 1 : 2) : 0);
}

}  // namespace dfl
