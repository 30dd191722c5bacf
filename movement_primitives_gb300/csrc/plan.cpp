// Host planner of the strided tile layout copy: validation, canonical forms,
// the kernel-class decision, the [outer, threads, vec] vector width and the
// shared-memory bank simulator that picks the warp permute's XOR swizzle.
//
// Everything here is integer host code run once per call (microseconds).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "lc_internal.h"

namespace lc {

namespace {

constexpr int kWarp = 32;
constexpr int64_t kMaxOffset = int64_t(1) << 62;  // byte offsets stay in int64
constexpr int64_t kBruteInjective = int64_t(1) << 24;

bool mul_ok(int64_t a, int64_t b, int64_t *r) { return !__builtin_mul_overflow(a, b, r); }
bool add_ok(int64_t a, int64_t b, int64_t *r) { return !__builtin_add_overflow(a, b, r); }

bool valid_width(int w) { return w == 1 || w == 2 || w == 4 || w == 8 || w == 16; }

// Neighbouring modes (outer, inner) merge when they are row-major contiguous
// on BOTH sides: s_outer == s_inner * e_inner and d_outer == d_inner * e_inner.
void coalesce(ModeList *ml) {
    int n = 0;
    for (int i = 0; i < ml->n; ++i) {
        const Mode &c = ml->m[i];
        if (n > 0) {
            Mode &o = ml->m[n - 1];
            if (o.s == c.s * c.e && o.d == c.d * c.e) {
                o.e *= c.e;
                o.s = c.s;
                o.d = c.d;
                continue;
            }
        }
        ml->m[n++] = c;
    }
    ml->n = n;
}

// Modes of a set are "dense" on one side when their offsets tile [0, prod e)
// exactly: sorted by that side's stride they read 1, e_a, e_a * e_b, ...
bool dense(const ModeList &ml, int first, bool src_side) {
    std::vector<std::pair<int64_t, int64_t>> v;  // (stride, extent)
    for (int i = first; i < ml.n; ++i)
        v.push_back({src_side ? ml.m[i].s : ml.m[i].d, ml.m[i].e});
    std::sort(v.begin(), v.end());
    int64_t expect = 1;
    for (auto &p : v) {
        if (p.first != expect) return false;
        expect *= p.second;
    }
    return true;
}

// Is  i -> sum_k i_k d_k  one-to-one over the modes (every d_k > 0)?
// Modes sorted by stride ascending; a split after the first p modes is
// proof-carrying when everything those modes reach is below G, the gcd of the
// remaining strides: an offset is then a + G b with a in [0, G) from the
// first p modes and b from the rest divided by G, a unique decomposition, so
// the whole map is one-to-one exactly when both parts are.  (A stride larger
// than everything the smaller modes reach is the case of a single remaining
// mode.)  Parts no split decides are enumerated up to kBruteInjective words;
// beyond that the question stays open (LC_ERR_UNDECIDED).
int64_t gcd64(int64_t a, int64_t b) {
    while (b) { const int64_t t = a % b; a = b; b = t; }
    return a;
}

int enumerate_injective(const std::vector<std::pair<int64_t, int64_t>> &v) {
    int64_t total = 1;
    for (auto &p : v) total *= p.second;
    if (total > kBruteInjective) return LC_ERR_UNDECIDED;
    std::vector<int64_t> offs;
    offs.reserve(size_t(total));
    std::vector<int64_t> idx(v.size(), 0);
    for (int64_t t = 0; t < total; ++t) {
        int64_t o = 0;
        for (size_t i = 0; i < v.size(); ++i) o += idx[i] * v[i].first;
        offs.push_back(o);
        for (size_t i = v.size(); i-- > 0;) {
            if (++idx[i] < v[i].second) break;
            idx[i] = 0;
        }
    }
    std::sort(offs.begin(), offs.end());
    return std::adjacent_find(offs.begin(), offs.end()) == offs.end() ? LC_OK : LC_ERR_NOT_INJECTIVE;
}

// v: (stride, extent) pairs sorted by stride ascending, every extent > 1.
int injective_sorted(const std::vector<std::pair<int64_t, int64_t>> &v) {
    if (v.size() <= 1) return LC_OK;
    // suffix gcds of the strides
    std::vector<int64_t> g(v.size() + 1, 0);
    for (size_t i = v.size(); i-- > 0;) g[i] = gcd64(v[i].first, g[i + 1]);
    int64_t reach = 0;
    for (size_t p = 1; p < v.size(); ++p) {
        reach += (v[p - 1].second - 1) * v[p - 1].first;
        if (reach < g[p]) {
            std::vector<std::pair<int64_t, int64_t>> lo(v.begin(), v.begin() + p), hi(v.begin() + p, v.end());
            for (auto &q : hi) q.first /= g[p];
            int st = injective_sorted(lo);
            if (st == LC_OK) st = injective_sorted(hi);
            return st;
        }
    }
    return enumerate_injective(v);
}

int dst_injective(const ModeList &ml) {
    std::vector<std::pair<int64_t, int64_t>> v;
    for (int i = 0; i < ml.n; ++i)
        if (ml.m[i].e > 1) v.push_back({ml.m[i].d, ml.m[i].e});
    std::sort(v.begin(), v.end());
    return injective_sorted(v);
}

int check_layout(const lc_tile_layout *l) {
    if (l->rank < 1 || l->rank > LC_MAX_RANK) return LC_ERR_RANK;
    for (int k = 0; k < l->rank; ++k)
        if (l->shape[k] < 0) return LC_ERR_SHAPE;
    if (l->offset < 0 || l->tile_stride < 0) return LC_ERR_BAD_STRIDE;
    return LC_OK;
}

// 1 + sum (e - 1) * stride, with overflow reported.
int cosize(const lc_tile_layout *l, int64_t *out) {
    int64_t c = 1;
    for (int k = 0; k < l->rank; ++k) {
        if (l->shape[k] == 0) { *out = 0; return LC_OK; }
        int64_t t;
        if (!mul_ok(l->shape[k] - 1, l->stride[k], &t) || !add_ok(c, t, &c)) return LC_ERR_OVERFLOW;
    }
    *out = c;
    return LC_OK;
}

// Byte address alignment of a base (pointer + offset * w).
uintptr_t base_addr(uintptr_t p, int64_t off, int w) { return p + uintptr_t(off) * uintptr_t(w); }

// --------------------------------------------------------------------------
// bank simulator
// --------------------------------------------------------------------------

// Worst degree of one warp-wide access: 128-byte wavefronts (32 lanes for
// words up to 4 bytes, 16 lanes for 8, 8 lanes for 16); per bank, the number
// of distinct 4-byte words it must deliver.
int access_degree(const int64_t *byte_addr, int w) {
    const int per = w <= 4 ? kWarp : 128 / w;
    int worst = 0;
    for (int g = 0; g < kWarp; g += per) {
        int64_t words[kWarp * 4];
        int nw = 0;
        for (int l = g; l < g + per; ++l) {
            int64_t first = byte_addr[l] >> 2, last = (byte_addr[l] + w - 1) >> 2;
            for (int64_t x = first; x <= last; ++x) words[nw++] = x;
        }
        std::sort(words, words + nw);
        nw = int(std::unique(words, words + nw) - words);
        int per_bank[32] = {0};
        for (int i = 0; i < nw; ++i) {
            int b = int(words[i] & 31);
            worst = std::max(worst, ++per_bank[b]);
        }
    }
    return worst;
}

int64_t unit_size(const ModeList &u) {
    int64_t t = 1;
    for (int i = 0; i < u.n; ++i) t *= u.m[i].e;
    return t;
}

}  // namespace

int access_degree_vec(const int64_t *byte_addr, int width) { return access_degree(byte_addr, width); }

bool mul_ok_ext(int64_t a, int64_t b, int64_t *r) { return !__builtin_mul_overflow(a, b, r); }
bool add_ok_ext(int64_t a, int64_t b, int64_t *r) { return !__builtin_add_overflow(a, b, r); }

FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d ? d : 1;
    int s = 0;
    while ((uint64_t(1) << s) < f.d) ++s;
    f.s = s;
    f.m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << s) - f.d)) / f.d + 1);
    return f;
}

void phase_degrees(const ModeList &unit, int w, int k, int shift, int *rd, int *wd) {
    const int64_t total = unit_size(unit);
    const int P = int(total / kWarp);
    const int mask = (1 << k) - 1;
    int r_worst = 0, w_worst = 0;
    for (int r = 0; r < P; ++r) {
        int64_t ra[kWarp], wa[kWarp];
        for (int lane = 0; lane < kWarp; ++lane) {
            const int j = r ^ ((lane >> shift) & mask);
            int64_t flat = lane + int64_t(kWarp) * j, so = 0, dof = 0;
            for (int i = unit.n - 1; i >= 0; --i) {
                const int64_t c = flat % unit.m[i].e;
                flat /= unit.m[i].e;
                so += c * unit.m[i].s;
                dof += c * unit.m[i].d;
            }
            ra[lane] = so * w;
            wa[lane] = dof * w;
        }
        r_worst = std::max(r_worst, access_degree(ra, w));
        w_worst = std::max(w_worst, access_degree(wa, w));
    }
    *rd = r_worst;
    *wd = w_worst;
}

int choose_xor(const ModeList &unit, int w, int *k_out, int *shift_out, int *rd_out, int *wd_out) {
    const int64_t P = unit_size(unit) / kWarp;
    int kmax = 0;
    if (P > 0 && (P & (P - 1)) == 0)
        while ((int64_t(1) << (kmax + 1)) <= P) ++kmax;
    int best = 1 << 30, bk = 0, bs = 0, brd = 0, bwd = 0;
    for (int k = 0; k <= kmax; ++k) {
        const int smax = k ? 5 - k : 0;
        for (int shift = 0; shift <= smax; ++shift) {
            int rd, wd;
            phase_degrees(unit, w, k, shift, &rd, &wd);
            if (rd <= 1 && wd <= 1) {
                *k_out = k; *shift_out = shift; *rd_out = rd; *wd_out = wd;
                return 0;
            }
            if (std::max(rd, wd) < best) {
                best = std::max(rd, wd); bk = k; bs = shift; brd = rd; bwd = wd;
            }
        }
    }
    *k_out = bk; *shift_out = bs; *rd_out = brd; *wd_out = bwd;
    return 1;
}

// Both copies of the shared-memory transpose, per warp instruction, on one
// tile of TX rows x RB bytes (smem_geometry), chunk k of row x stored in
// slot k ^ ((x >> shift) & mask).  Copy 1: thread t of 256 moves chunk
// t % NC of row t / NC (+ 256 / NC per round), C bytes.  Copy 2: lanes read
// word y of 32 consecutive rows; word y of row x starts at byte e + y * w of
// the row's chunk sequence (e = the row's lead-in, taken as 0: rows with
// different lead-ins may meet in a bank at most twice).
SmemSwizzle choose_smem_swizzle(int w) {
    const SmemGeo g = smem_geometry(w);
    const int nc = g.RB / g.C;
    SmemSwizzle best;
    int best_deg = 1 << 30;
    for (int k = 0; (1 << k) <= nc; ++k) {
        for (int shift = 0; shift <= (k ? 6 - k : 0); ++shift) {
            const int mask = (1 << k) - 1;
            auto sw = [&](int x) { return (x >> shift) & mask; };
            int rd = 0, wd = 0;
            for (int r = 0; r < g.TX * nc / 256; ++r) {
                for (int t0 = 0; t0 < 256; t0 += kWarp) {
                    int64_t ad[kWarp];
                    for (int l = 0; l < kWarp; ++l) {
                        const int t = t0 + l, x = t / nc + r * (256 / nc), c = t % nc;
                        ad[l] = int64_t(x) * g.RB + int64_t(c ^ sw(x)) * g.C;
                    }
                    wd = std::max(wd, access_degree(ad, g.C));
                }
            }
            for (int y = 0; y < g.TYW; ++y) {
                for (int base = 0; base < g.TX; base += kWarp) {
                    int64_t ad[kWarp];
                    for (int l = 0; l < kWarp; ++l) {
                        const int x = base + l;
                        ad[l] = int64_t(x) * g.RB + ((int64_t(y) * w) ^ (int64_t(sw(x)) * g.C));
                    }
                    rd = std::max(rd, access_degree(ad, w));
                }
            }
            const int deg = std::max(rd, wd);
            if (deg < best_deg) {
                best_deg = deg;
                best.shift = shift;
                best.mask = mask;
                best.cr = rd;
                best.cw = wd;
            }
            if (deg <= 1) return best;
        }
    }
    return best;
}

int align_shards(const lc_tile_layout *src, const lc_tile_layout *dst, ModeList *out) {
    int st;
    if ((st = check_layout(src)) || (st = check_layout(dst))) return st;
    int ns = 0, nd = 0;
    Mode tmp[LC_MAX_RANK];
    int64_t de[LC_MAX_RANK], dd[LC_MAX_RANK];
    for (int k = 0; k < dst->rank; ++k)
        if (dst->shape[k] != 1) { de[nd] = dst->shape[k]; dd[nd] = dst->stride[k]; ++nd; }
    for (int k = 0; k < src->rank; ++k)
        if (src->shape[k] != 1) { tmp[ns] = Mode{src->shape[k], src->stride[k], 0}; ++ns; }
    if (ns != nd) return LC_ERR_EXTENT_MISMATCH;
    out->n = 0;
    for (int i = 0; i < ns; ++i) {
        if (tmp[i].e != de[i]) return LC_ERR_EXTENT_MISMATCH;
        out->m[out->n++] = Mode{tmp[i].e, tmp[i].s, dd[i]};
    }
    coalesce(out);
    return LC_OK;
}

// --------------------------------------------------------------------------
// the plan
// --------------------------------------------------------------------------

namespace {

// Widest vector (16, 8, 4, 2, 1 bytes, at least one word) whose per-thread
// pointers all stay aligned ("copy -> gmem_smem", section "Algorithm",
// step 2): the run length is a multiple of it, so are every other stride on
// both sides and both base offsets, and so are the two base addresses.
int choose_vec(const Plan &p, const PtrInfo &ptr) {
    for (int bytes = 16; bytes >= p.w; bytes >>= 1) {
        if (bytes % p.w) continue;
        const int v = bytes / p.w;
        if (v == 1) return 1;
        if (p.vec.run % v) continue;
        bool ok = p.src_off % v == 0 && p.dst_off % v == 0;
        for (int i = 0; ok && i < p.vec.outer.n; ++i)
            ok = p.vec.outer.m[i].s % v == 0 && p.vec.outer.m[i].d % v == 0;
        if (ok && ptr.check)
            ok = base_addr(ptr.src, p.src_off, p.w) % bytes == 0 &&
                 base_addr(ptr.dst, p.dst_off, p.w) % bytes == 0;
        if (ok) return v;
    }
    return 1;
}

void plan_vec(Plan *p, const PtrInfo &ptr) {
    p->vec = VecPlan{};
    const ModeList &sl = p->sorted;
    int n = sl.n;
    if (n > 0 && sl.m[n - 1].s == 1 && sl.m[n - 1].d == 1) {
        p->vec.run = sl.m[n - 1].e;
        --n;
    }
    for (int i = 0; i < n; ++i) p->vec.outer.m[i] = sl.m[i];
    p->vec.outer.n = n;
    p->vec.vec = choose_vec(*p, ptr);
}

constexpr int64_t kStageTarget = 4 * 1024;  // bytes of units one warp stages at once
constexpr int64_t kSmallAutoBytes = 32 * 1024;  // single tiles up to this size skip the warp classes
constexpr int64_t kSmallPlaneBytes = 16 * 1024;  // transposed planes up to this size prefer shared memory to TMA

// Warp permute: the smallest innermost (logical-order) mode suffix that is a
// dense block on both sides and a whole number of warp lanes (32 * P words,
// P <= 32); the rest of the modes enumerate units.  Units move whole with
// bulk copies, so their bytes and every unit base must be 16-byte aligned.
bool plan_warp(Plan *p, const PtrInfo &ptr, bool need_conflict_free) {
    const ModeList &lg = p->logical;
    const int w = p->w;  // unfused (caller guarantees p->fused == 1)
    int first = -1;
    int64_t U = 1;
    for (int i = lg.n - 1; i >= 0; --i) {
        U *= lg.m[i].e;
        if (U > 32 * kWarp) break;
        if (U % kWarp == 0 && dense(lg, i, true) && dense(lg, i, false)) { first = i; break; }
    }
    if (first < 0 || lg.n - first > LC_MAX_RANK) return false;
    if ((U * w) % 16) return false;
    for (int i = 0; i < first; ++i)
        if ((lg.m[i].s * w) % 16 || (lg.m[i].d * w) % 16) return false;
    if ((p->src_off * w) % 16 || (p->dst_off * w) % 16) return false;
    if (ptr.check && (ptr.src % 16 || ptr.dst % 16)) return false;

    WarpPlan &wp = p->warp;
    wp = WarpPlan{};
    for (int i = first; i < lg.n; ++i) wp.unit.m[wp.unit.n++] = lg.m[i];
    for (int i = 0; i < first; ++i) wp.batch.m[wp.batch.n++] = lg.m[i];
    wp.U = U;
    wp.P = int(U / kWarp);
    const int bad = choose_xor(wp.unit, w, &wp.k, &wp.shift, &wp.cr, &wp.cw);
    if (bad && need_conflict_free) return false;
    wp.mask = (1 << wp.k) - 1;
    wp.n_units = p->total / U;
    wp.units_per_stage = std::max<int64_t>(1, std::min<int64_t>(wp.n_units, kStageTarget / (U * w)));
    return true;
}

// Warp-shuffle permute: X = the mode contiguous in dst, Y = the mode
// contiguous in src.  One of them spans exactly V = 16 / w words and the
// other a multiple of V, so that every V x V block has its rows as 16-byte
// source chunks and its columns as 16-byte destination chunks:
//   X.e == V (the page's (4, 32) -> strides (1, 4) case): block k of a batch
//     entry holds columns k V .. k V + V - 1 of Y; lane a reads row a
//     (source a X.s + k V) and writes column k V + a (destination
//     (k V + a) Y.d);
//   Y.e == V (its mirror): block k holds rows k V .. k V + V - 1 of X; lane
//     a reads row k V + a (source (k V + a) X.s) and writes column a
//     (destination a Y.d + k V).
// Every chunk must be 16-byte aligned: X.s and Y.d multiples of V, every
// batch stride and both base offsets multiples of 16 bytes.
bool plan_shuffle(Plan *p, const PtrInfo &ptr) {
    const ModeList &sl = p->sorted;
    const int w = p->w;
    if (w > 8) return false;
    const int64_t V = 16 / w;
    int xi = -1, yi = -1;
    for (int i = 0; i < sl.n; ++i) {
        if (sl.m[i].d == 1) xi = i;
        if (sl.m[i].s == 1) yi = i;
    }
    if (xi < 0 || yi < 0 || xi == yi) return false;
    const Mode X = sl.m[xi], Y = sl.m[yi];
    if (X.s % V || Y.d % V) return false;
    ShflPlan &sp = p->shfl;
    sp = ShflPlan{};
    sp.V = int(V);
    if (X.e == V && Y.e % V == 0) {
        sp.kb = Y.e / V;
        sp.sa = X.s;
        sp.sk = V;
        sp.da = Y.d;
        sp.dk = V * Y.d;
    } else if (Y.e == V && X.e % V == 0) {
        sp.kb = X.e / V;
        sp.sa = X.s;
        sp.sk = V * X.s;
        sp.da = Y.d;
        sp.dk = V;
    } else {
        return false;
    }
    int64_t n_batch = 1;
    for (int i = 0; i < sl.n; ++i) {
        if (i == xi || i == yi) continue;
        const Mode &b = sl.m[i];
        if ((b.s * w) % 16 || (b.d * w) % 16 || b.e >= (int64_t(1) << 31)) return false;
        sp.batch.m[sp.batch.n++] = b;
        n_batch *= b.e;
    }
    if ((p->src_off * w) % 16 || (p->dst_off * w) % 16) return false;
    if (ptr.check && (ptr.src % 16 || ptr.dst % 16)) return false;
    if (sp.kb >= (int64_t(1) << 31) || n_batch >= (int64_t(1) << 31)) return false;
    sp.n_blocks = n_batch * sp.kb;
    if (sp.n_blocks >= (int64_t(1) << 31)) return false;
    return true;
}

// Tile transpose: a mode contiguous in dst (X) and another contiguous in src
// (Y); at most three other (batch) modes; TMA needs 16-byte aligned bases
// and 16-byte multiple strides, stores need the same on the destination.
bool plan_tile(Plan *p, const PtrInfo &ptr) {
    const ModeList &sl = p->sorted;
    int xi = -1, yi = -1;
    for (int i = 0; i < sl.n; ++i) {
        if (sl.m[i].d == 1) xi = i;
        if (sl.m[i].s == 1) yi = i;
    }
    if (xi < 0 || yi < 0 || xi == yi) return false;
    TilePlan &tp = p->tile;
    tp = TilePlan{};
    tp.X = sl.m[xi];
    tp.Y = sl.m[yi];
    for (int i = 0; i < sl.n; ++i)
        if (i != xi && i != yi) tp.batch.m[tp.batch.n++] = sl.m[i];
    if (tp.batch.n > 3) return false;
    const int w = p->w;
    auto a16 = [](int64_t x) { return x % 16 == 0; };
    if (!a16(tp.X.s * w) || !a16(tp.Y.d * w)) return false;
    if (tp.X.s * w >= (int64_t(1) << 40)) return false;
    for (int i = 0; i < tp.batch.n; ++i) {
        const Mode &b = tp.batch.m[i];
        if (b.s <= 0 || !a16(b.s * w) || !a16(b.d * w)) return false;
        if (b.s * w >= (int64_t(1) << 40) || b.e > (int64_t(1) << 31)) return false;
    }
    if (tp.X.e > (int64_t(1) << 31) || tp.Y.e * (w == 16 ? 2 : 1) > (int64_t(1) << 31)) return false;
    if (!a16(p->src_off * w) || !a16(p->dst_off * w)) return false;
    if (ptr.check && (ptr.src % 16 || ptr.dst % 16)) return false;
    if (tile_direct_geometry(w, p->total * w, tp.X.e, tp.Y.e, &tp.R, &tp.TY, &tp.threads)) {
        tp.S = 0;
        tp.direct = 1;
    } else if (ptr.no_tma) {
        return false;  // the other forms load through TMA tensor maps
    } else if (tile_tstore_geometry(w, p->total * w, tp.X.e, tp.Y.d * w, &tp.R, &tp.TY, &tp.S, &tp.threads)) {
        tp.tstore = 1;
    } else {
        tile_geometry(w, p->total * w, &tp.R, &tp.TY, &tp.S, &tp.threads);  // the kernel's per-width table
    }
    return true;
}

// Shared-memory transpose: a mode contiguous in dst (X) and another in src
// (Y), any number of batch modes, any alignment beyond the word size.
bool plan_smem(Plan *p) {
    const ModeList &sl = p->sorted;
    int xi = -1, yi = -1;
    for (int i = 0; i < sl.n; ++i) {
        if (sl.m[i].d == 1) xi = i;
        if (sl.m[i].s == 1) yi = i;
    }
    if (xi < 0 || yi < 0 || xi == yi) return false;
    TilePlan &tp = p->tile;
    tp = TilePlan{};
    tp.X = sl.m[xi];
    tp.Y = sl.m[yi];
    for (int i = 0; i < sl.n; ++i)
        if (i != xi && i != yi) tp.batch.m[tp.batch.n++] = sl.m[i];
    const SmemGeo g = smem_geometry(p->w);
    tp.R = g.TX;
    tp.TY = g.TYW;
    tp.S = 1;
    tp.threads = 256;
    // the kernel decodes tile indices in 32 bits
    int64_t n_tiles = ((tp.X.e + tp.R - 1) / tp.R) * ((tp.Y.e + tp.TY - 1) / tp.TY);
    for (int i = 0; i < tp.batch.n; ++i) n_tiles *= tp.batch.m[i].e;
    if (n_tiles >= (int64_t(1) << 31)) return false;
    p->smem_swz = choose_smem_swizzle(p->w);
    return true;
}

// TMA tensor copy: the innermost destination-ordered mode is contiguous on
// both sides; the modes, innermost first, become the dimensions of a source
// and a destination tensor map.  The box grows from the innermost dimension
// outwards (at most 256 per dimension) while the tile stays within
// kTmaTileBytes.
#ifndef LC_TMA_MIN_RUN_BYTES
#define LC_TMA_MIN_RUN_BYTES 64
#endif
// Box split between the destination's and the source's next contiguous modes
// for runs shorter than this many bytes (measured on GB300: head permutes
// with 64- and 128-byte runs gain 16 % and 9 %; 256-byte runs lose 2-3 %).
#ifndef LC_TMA_BALANCE_BELOW
#define LC_TMA_BALANCE_BELOW 256
#endif
constexpr int64_t kTmaMinRunBytes = LC_TMA_MIN_RUN_BYTES;
constexpr int64_t kTmaTileBytes = LC_TMA_TILE_BYTES;

bool plan_tma(Plan *p, const PtrInfo &ptr) {
    if (ptr.no_tma) return false;
    const ModeList &sl = p->sorted;
    const int w = p->w;
    if (sl.n < 2 || sl.n > 5) return false;
    const Mode &in = sl.m[sl.n - 1];
    if (in.s != 1 || in.d != 1) return false;
    if ((in.e * w) % 16 || in.e * w < kTmaMinRunBytes) return false;
    const int mult = w == 16 ? 2 : 1;  // 16-byte words travel as two 8-byte elements
    const int eb = w / mult;
    if (in.e * mult >= (int64_t(1) << 31)) return false;
    for (int i = 0; i + 1 < sl.n; ++i) {
        const Mode &m = sl.m[i];
        if (m.s <= 0 || m.d <= 0 || (m.s * w) % 16 || (m.d * w) % 16) return false;
        if (m.s * w >= (int64_t(1) << 40) || m.d * w >= (int64_t(1) << 40) || m.e >= (int64_t(1) << 31)) return false;
    }
    if ((p->src_off * w) % 16 || (p->dst_off * w) % 16) return false;
    if (ptr.check && (ptr.src % 16 || ptr.dst % 16)) return false;
    TmaPlan &tp = p->tma;
    tp = TmaPlan{};
    tp.rank = sl.n;
    int64_t dims[5];
    for (int k = 0; k < sl.n; ++k) dims[k] = sl.m[sl.n - 1 - k].e * (k == 0 ? mult : 1);
    tp.box[0] = static_cast<int>(std::min<int64_t>(dims[0], 256));
    int64_t bytes = int64_t(tp.box[0]) * eb;
    for (int k = 1; k < sl.n; ++k) tp.box[k] = 1;
    // Dimension 1 continues the run on the destination side; the dimension
    // whose source stride equals the run continues it on the source side.
    // When they differ and runs are short, the box splits its budget between
    // the two, so that both sides move segments of several runs instead of
    // one side moving isolated runs.
    int ksrc = -1;
    if (tp.box[0] == dims[0])
        for (int k = 2; k < sl.n; ++k)
            if (sl.m[sl.n - 1 - k].s == in.e) { ksrc = k; break; }
    const int64_t budget = std::max<int64_t>(1, kTmaTileBytes / bytes);
    if (ksrc > 1 && int64_t(tp.box[0]) * eb < LC_TMA_BALANCE_BELOW) {
        int64_t bs = 1;
        while ((bs * 2) * (bs * 2) <= budget) bs *= 2;
        bs = std::min<int64_t>({bs, dims[ksrc], 256});
        const int64_t b1 = std::max<int64_t>(1, std::min<int64_t>({dims[1], 256, budget / bs}));
        bs = std::max<int64_t>(1, std::min<int64_t>({dims[ksrc], 256, budget / b1}));
        tp.box[1] = static_cast<int>(b1);
        tp.box[ksrc] = static_cast<int>(bs);
        bytes *= b1 * bs;
    } else {
        for (int k = 1; k < sl.n; ++k) {
            const int64_t b = std::max<int64_t>(1, std::min<int64_t>({dims[k], 256, kTmaTileBytes / bytes}));
            tp.box[k] = static_cast<int>(b);
            bytes *= b;
        }
    }
    uint64_t n_tiles = 1;
    for (int k = 0; k < sl.n; ++k) n_tiles *= uint64_t((dims[k] + tp.box[k] - 1) / tp.box[k]);
    if (n_tiles >= (uint64_t(1) << 32)) return false;
    tp.stage_bytes = bytes;
    p->tile = TilePlan{};
    p->tile.R = tp.box[1];
    p->tile.TY = tp.box[0];
    p->tile.S = LC_TMA_STAGES;
    p->tile.threads = 32;
    return true;
}

// A contiguous run of L words with L * w <= 16 bytes (a power of two) moves
// as one wider word when every other stride, both offsets and both base
// addresses allow it: the copy is then a permute of (L * w)-byte words.
void fuse_inner_run(Plan *p, const PtrInfo &ptr) {
    ModeList &sl = p->sorted;
    if (sl.n == 0) return;
    const Mode r = sl.m[sl.n - 1];
    if (r.s != 1 || r.d != 1) return;
    const int64_t L = r.e;
    const int64_t nb = L * p->w;
    if (nb > 16 || (nb & (nb - 1))) return;
    if (p->src_off % L || p->dst_off % L) return;
    for (int i = 0; i + 1 < sl.n; ++i)
        if (sl.m[i].s % L || sl.m[i].d % L) return;
    if (ptr.check && (base_addr(ptr.src, p->src_off, p->w) % nb ||
                      base_addr(ptr.dst, p->dst_off, p->w) % nb))
        return;
    --sl.n;
    for (int i = 0; i < sl.n; ++i) { sl.m[i].s /= L; sl.m[i].d /= L; }
    p->src_off /= L;
    p->dst_off /= L;
    p->w = int(nb);
    p->fused = int(L);
}

}  // namespace

namespace {

// Validation and planning.  `ptr` carries only the two base addresses modulo
// 16 (every alignment decision depends on nothing more); NULL, alignment and
// overlap of the real pointers are checked by make_plan.
int make_plan_core(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w,
                   int64_t n_tiles, int32_t kernel, const PtrInfo &ptr, Plan *out) {
    if (!src || !dst || !out) return LC_ERR_NULL;
    int st;
    if ((st = check_layout(src)) || (st = check_layout(dst))) return st;
    if (!valid_width(w)) return LC_ERR_ELEM_BYTES;
    if (n_tiles < 0) return LC_ERR_SHAPE;
    if (kernel < LC_KERNEL_AUTO || kernel > LC_KERNEL_SMEM_STAGED) return LC_ERR_UNSUPPORTED;

    Plan p;
    p.w = w;
    // pair the non-unit modes ("equal non-unit extents")
    ModeList paired;
    if ((st = align_shards(src, dst, &paired))) return st;
    // align_shards already coalesced; recount the total from the raw extents
    int64_t total = n_tiles;
    for (int k = 0; k < src->rank; ++k)
        if (!mul_ok(total, src->shape[k], &total)) return LC_ERR_OVERFLOW;
    p.total = total;
    if (total == 0) { p.kernel = kernel ? kernel : LC_KERNEL_VEC_COPY; *out = p; return LC_OK; }

    for (int k = 0; k < src->rank; ++k)
        if (src->shape[k] != 1 && src->stride[k] < 0) return LC_ERR_BAD_STRIDE;
    for (int k = 0; k < dst->rank; ++k)
        if (dst->shape[k] != 1 && dst->stride[k] <= 0) return LC_ERR_BAD_STRIDE;

    int64_t cs, cd;
    if ((st = cosize(src, &cs)) || (st = cosize(dst, &cd))) return st;
    const int64_t sts = src->tile_stride ? src->tile_stride : cs;
    const int64_t dts = dst->tile_stride ? dst->tile_stride : cd;

    // largest offsets reached, which must stay addressable in bytes
    int64_t smax, dmax, t;
    if (!mul_ok(n_tiles - 1, sts, &t) || !add_ok(t, src->offset + cs - 1, &smax)) return LC_ERR_OVERFLOW;
    if (!mul_ok(n_tiles - 1, dts, &t) || !add_ok(t, dst->offset + cd - 1, &dmax)) return LC_ERR_OVERFLOW;
    if (smax >= kMaxOffset / 16 || dmax >= kMaxOffset / 16) return LC_ERR_OVERFLOW;

    // logical order: the tile mode outermost, then the paired modes, merged
    ModeList lg;
    if (n_tiles > 1) lg.m[lg.n++] = Mode{n_tiles, sts, dts};
    for (int i = 0; i < paired.n; ++i) lg.m[lg.n++] = paired.m[i];
    coalesce(&lg);
    if ((st = dst_injective(lg))) return st;

    p.src_lo = src->offset * w;
    p.src_hi = (smax + 1) * w;
    p.dst_lo = dst->offset * w;
    p.dst_hi = (dmax + 1) * w;
    p.logical = lg;
    p.src_off = src->offset;
    p.dst_off = dst->offset;
    // destination order: stride descending (stable), merged again
    p.sorted = lg;
    std::stable_sort(p.sorted.m, p.sorted.m + p.sorted.n,
                     [](const Mode &a, const Mode &b) { return a.d > b.d; });
    coalesce(&p.sorted);

    p.src_l = *src;
    p.dst_l = *dst;
    p.n_tiles = n_tiles;
    if (kernel == LC_KERNEL_SMEM_STAGED) {
        int64_t N = 1;
        for (int k = 0; k < src->rank; ++k) N *= src->shape[k];
        if (N * w > LC_STAGED_MAX_BYTES) return LC_ERR_UNSUPPORTED;
        plan_vec(&p, ptr);
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }
    if (kernel == LC_KERNEL_WARP_PERMUTE) {
        plan_vec(&p, ptr);
        if (!plan_warp(&p, ptr, false)) return LC_ERR_UNSUPPORTED;
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }
    fuse_inner_run(&p, ptr);
    plan_vec(&p, ptr);  // always available: the fallback of every other class
    if (kernel == LC_KERNEL_WARP_SHUFFLE) {
        if (!plan_shuffle(&p, ptr)) return LC_ERR_UNSUPPORTED;
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }
    if (kernel == LC_KERNEL_TILE_TRANSPOSE) {
        if (!plan_tile(&p, ptr)) return LC_ERR_UNSUPPORTED;
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }
    if (kernel == LC_KERNEL_SMEM_TRANSPOSE) {
        if (!plan_smem(&p)) return LC_ERR_UNSUPPORTED;
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }
    if (kernel == LC_KERNEL_TMA_COPY) {
        if (!plan_tma(&p, ptr)) return LC_ERR_UNSUPPORTED;
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }
    if (kernel == LC_KERNEL_VEC_COPY) {
        p.kernel = kernel;
        *out = p;
        return LC_OK;
    }

    // automatic choice
    const ModeList &sl = p.sorted;
    const bool run = sl.n > 0 && sl.m[sl.n - 1].s == 1 && sl.m[sl.n - 1].d == 1;
    bool has_x = false, has_y = false;
    for (int i = 0; i < sl.n; ++i) { has_x |= sl.m[i].d == 1; has_y |= sl.m[i].s == 1; }
    // A single small tile is a few CTAs' work at most: the warp classes would
    // give it one or two warps and the staged copy one CTA.  Measured per copy
    // replayed from a graph (32 KiB and less): the shared-memory transpose is
    // fastest for words of 4 bytes and more (the page's 32 x 32 fp32
    // transpose: 1.9 us, staged 2.6, tile 2.2), the tile transpose for 1- and
    // 2-byte words (a 128 x 256 byte transpose: 2.1 us, shared-memory
    // transpose 3.5, staged 40), the vector copy where neither of those
    // plans (a 37 x 55 2-byte transpose: 2.0 us, shared-memory transpose 2.8).
    if (n_tiles == 1 && total * w <= kSmallAutoBytes && !run) {
        if (has_x && has_y) {
            Plan q = p;
            if (w >= 4 && plan_smem(&q)) { q.kernel = LC_KERNEL_SMEM_TRANSPOSE; *out = q; return LC_OK; }
            q = p;
            if (plan_tile(&q, ptr)) { q.kernel = LC_KERNEL_TILE_TRANSPOSE; *out = q; return LC_OK; }
        }
        p.kernel = LC_KERNEL_VEC_COPY;
        *out = p;
        return LC_OK;
    }
    if (!run && has_x && has_y) {
        if (plan_shuffle(&p, ptr)) { p.kernel = LC_KERNEL_WARP_SHUFFLE; *out = p; return LC_OK; }
        // 16-byte words past 8 a lane hold 128 registers of words and spill:
        // a batch of 32 x 32 of them moved 34 % of the copy peak on the warp
        // permute and 100 % on the shared-memory transpose
        if (p.fused == 1) {
            Plan q = p;
            if (plan_warp(&q, ptr, true) && !(q.w == 16 && q.warp.P > 8)) {
                q.kernel = LC_KERNEL_WARP_PERMUTE;
                *out = q;
                return LC_OK;
            }
        }
        Plan q = p;
        if (plan_tile(&q, ptr)) {
            // batches of small planes of wide words: the TMA tile's boxes
            // cover little of each plane; measured on batches of 32 x 32 planes,
            // 8-byte words 44.9 against 38.2 %, 16-byte 100.3 against 37.9,
            // and 64 x 32 of 4-byte words 44.4 against 39.0
            Plan r = p;
            if (q.w >= 4 && q.tile.X.e * q.tile.Y.e * q.w <= kSmallPlaneBytes && plan_smem(&r)) {
                r.kernel = LC_KERNEL_SMEM_TRANSPOSE;
                *out = r;
                return LC_OK;
            }
            q.kernel = LC_KERNEL_TILE_TRANSPOSE;
            *out = q;
            return LC_OK;
        }
        if (plan_smem(&p)) { p.kernel = LC_KERNEL_SMEM_TRANSPOSE; *out = p; return LC_OK; }
    }
    if (run && plan_tma(&p, ptr)) { p.kernel = LC_KERNEL_TMA_COPY; *out = p; return LC_OK; }
    p.kernel = LC_KERNEL_VEC_COPY;
    *out = p;
    return LC_OK;
}

// Plans are pure functions of (layouts, width, tiles, kernel, base addresses
// mod 16); a small cache keeps the bank simulator off the per-call path.
std::mutex g_cache_mu;
std::unordered_map<std::string, Plan> g_cache;
constexpr size_t kCacheMax = 512;

void append(std::string &k, const void *p, size_t n) { k.append(static_cast<const char *>(p), n); }

std::string cache_key(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w, int64_t n_tiles,
                      int32_t kernel, const PtrInfo &ptr) {
    std::string k;
    for (const lc_tile_layout *l : {src, dst}) {
        append(k, &l->rank, sizeof(l->rank));
        append(k, l->shape, sizeof(int64_t) * size_t(l->rank));
        append(k, l->stride, sizeof(int64_t) * size_t(l->rank));
        append(k, &l->offset, sizeof(l->offset));
        append(k, &l->tile_stride, sizeof(l->tile_stride));
    }
    const int64_t tail[4] = {w, n_tiles, kernel,
                             int64_t((ptr.src & 15) | ((ptr.dst & 15) << 4) | (ptr.no_tma ? 256 : 0))};
    append(k, tail, sizeof(tail));
    return k;
}

int cached_plan(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w, int64_t n_tiles,
                int32_t kernel, const PtrInfo &mod, Plan *out) {
    const std::string key = cache_key(src, dst, w, n_tiles, kernel, mod);
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) { *out = it->second; return LC_OK; }
    }
    const int st = make_plan_core(src, dst, w, n_tiles, kernel, mod, out);
    if (st) return st;
    std::lock_guard<std::mutex> lk(g_cache_mu);
    if (g_cache.size() >= kCacheMax) g_cache.clear();
    g_cache.emplace(key, *out);
    return LC_OK;
}

// An exact in-place permute of dense units: every unit's source bytes are its
// destination bytes (same base address, equal batch strides).  The warp
// permute reads a whole group of units into its warp's shared slot before
// writing any of it back and groups are disjoint, so aliasing is safe
// ("permute_layout": a barrier between the phases makes aliasing safe).
bool exact_unit_alias(const Plan &p, const PtrInfo &ptr) {
    if (p.kernel != LC_KERNEL_WARP_PERMUTE) return false;
    if (ptr.src + uintptr_t(p.src_off * p.w) != ptr.dst + uintptr_t(p.dst_off * p.w)) return false;
    for (int i = 0; i < p.warp.batch.n; ++i)
        if (p.warp.batch.m[i].s != p.warp.batch.m[i].d) return false;
    return true;
}

}  // namespace

int make_plan(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w,
              int64_t n_tiles, int32_t kernel, const PtrInfo &ptr, Plan *out) {
    if (!src || !dst || !out) return LC_ERR_NULL;
    if (src->rank < 1 || src->rank > LC_MAX_RANK || dst->rank < 1 || dst->rank > LC_MAX_RANK)
        return LC_ERR_RANK;
    PtrInfo mod;
    mod.src = ptr.check ? (ptr.src & 15) : 0;
    mod.dst = ptr.check ? (ptr.dst & 15) : 0;
    mod.check = true;
    mod.no_tma = ptr.no_tma;
    int st = cached_plan(src, dst, w, n_tiles, kernel, mod, out);
    if (st) return st;
    if (!ptr.check || out->total == 0) return LC_OK;
    if (!ptr.src || !ptr.dst) return LC_ERR_NULL;
    if (ptr.src % uintptr_t(w) || ptr.dst % uintptr_t(w)) return LC_ERR_ALIGN;
    const uintptr_t s0 = ptr.src + uintptr_t(out->src_lo), s1 = ptr.src + uintptr_t(out->src_hi);
    const uintptr_t d0 = ptr.dst + uintptr_t(out->dst_lo), d1 = ptr.dst + uintptr_t(out->dst_hi);
    if (!(s0 < d1 && d0 < s1)) return LC_OK;
    // overlapping ranges: only the exact in-place unit permute is allowed
    if (kernel != LC_KERNEL_AUTO && kernel != LC_KERNEL_WARP_PERMUTE) return LC_ERR_OVERLAP;
    if (out->kernel != LC_KERNEL_WARP_PERMUTE) {
        Plan q;
        if (cached_plan(src, dst, w, n_tiles, LC_KERNEL_WARP_PERMUTE, mod, &q) != LC_OK) return LC_ERR_OVERLAP;
        *out = q;
    }
    return exact_unit_alias(*out, ptr) ? LC_OK : LC_ERR_OVERLAP;
}

void fill_info(const Plan &p, lc_plan_info *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = p.kernel;
    info->elem_bytes = p.w;
    info->total = p.total;
    const ModeList &ml = p.kernel == LC_KERNEL_WARP_PERMUTE ? p.logical : p.sorted;
    info->n_modes = ml.n;
    for (int i = 0; i < ml.n; ++i) {
        info->extent[i] = ml.m[i].e;
        info->src_stride[i] = ml.m[i].s;
        info->dst_stride[i] = ml.m[i].d;
    }
    info->vec = p.vec.vec;
    info->run = p.vec.run;
    info->unit_modes = p.warp.unit.n;
    info->P = p.warp.P;
    info->k = p.warp.k;
    info->shift = p.warp.shift;
    info->mask = p.warp.mask;
    info->conflicts_read = p.warp.cr;
    info->conflicts_write = p.warp.cw;
    info->units_per_chunk = p.warp.units_per_stage;
    info->tile_rows = p.tile.R;
    info->tile_cols = p.tile.TY;
    info->stages = p.tile.S;
    if (p.kernel == LC_KERNEL_TILE_TRANSPOSE) info->tile_form = p.tile.direct ? 1 : p.tile.tstore ? 2 : 0;
    if (p.kernel == LC_KERNEL_WARP_SHUFFLE) {  // V words per lane chunk, blocks per batch entry
        info->vec = p.shfl.V;
        info->P = p.shfl.V;
        info->units_per_chunk = p.shfl.kb;
    }
    if (p.kernel == LC_KERNEL_SMEM_TRANSPOSE) {
        int k = 0;
        while ((1 << k) - 1 < p.smem_swz.mask) ++k;
        info->k = k;
        info->shift = p.smem_swz.shift;
        info->mask = p.smem_swz.mask;
        info->conflicts_read = p.smem_swz.cr;
        info->conflicts_write = p.smem_swz.cw;
    }
}

// --------------------------------------------------------------------------
// loop-layout override (TileLang "loop_mapping.py": a loop_layout= annotation
// replaces the default plan)
// --------------------------------------------------------------------------

// Validates an override of n points: extents multiplying to n, each non-unit
// mode feeding exactly one of thread and slot, and each part a mixed radix
// once sorted by stride (exact partition of [0, T) x [0, L)).
int check_loop(const lc_loop_layout *loop, int64_t n, LoopPlan *out) {
    if (!loop || !out) return LC_ERR_NULL;
    if (loop->rank < 1 || loop->rank > LC_MAX_RANK) return LC_ERR_RANK;
    if (n < 0) return LC_ERR_SHAPE;
    int64_t prod = 1;
    for (int k = 0; k < loop->rank; ++k) {
        if (loop->shape[k] < 0) return LC_ERR_SHAPE;
        if (loop->thread_stride[k] < 0 || loop->slot_stride[k] < 0) return LC_ERR_BAD_STRIDE;
        if (!mul_ok(prod, loop->shape[k], &prod)) return LC_ERR_SHAPE;
    }
    if (prod != n) return LC_ERR_SHAPE;
    out->nt = out->ns = 0;
    out->T = out->L = 0;
    out->inner_run = 1;
    if (n == 0) return LC_OK;
    struct Part {
        int64_t e, stride, weight;
    };
    Part th[LC_MAX_RANK], sl[LC_MAX_RANK];
    int nt = 0, ns = 0;
    int64_t weight = 1;
    bool innermost = true;
    for (int k = loop->rank - 1; k >= 0; weight *= loop->shape[k], --k) {
        const int64_t e = loop->shape[k], ts = loop->thread_stride[k], ss = loop->slot_stride[k];
        if (e == 1) continue;
        if ((ts > 0) == (ss > 0)) return LC_ERR_BAD_STRIDE;
        if (ts > 0) th[nt++] = Part{e, ts, weight};
        else sl[ns++] = Part{e, ss, weight};
        if (innermost && ss == 1) out->inner_run = e;
        innermost = false;
    }
    auto by_stride = [](const Part &a, const Part &b) { return a.stride < b.stride; };
    std::stable_sort(th, th + nt, by_stride);
    std::stable_sort(sl, sl + ns, by_stride);
    int64_t T = 1, L = 1;
    for (int i = 0; i < nt; ++i) {
        if (th[i].stride != T) return LC_ERR_LOOP_LAYOUT;
        T *= th[i].e;
        if (T > LC_LOOP_MAX_THREADS) return LC_ERR_LOOP_LAYOUT;
        out->td[i] = LoopDigit{th[i].e, th[i].weight};
    }
    for (int i = 0; i < ns; ++i) {
        if (sl[i].stride != L) return LC_ERR_LOOP_LAYOUT;
        L *= sl[i].e;  // T * L == n, so no overflow
        out->sd[i] = LoopDigit{sl[i].e, sl[i].weight};
    }
    out->nt = nt;
    out->ns = ns;
    out->T = T;
    out->L = L;
    return LC_OK;
}

int make_loop_plan(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w, int64_t n_tiles,
                   const lc_loop_layout *loop, const PtrInfo &ptr, LoopPlan *out) {
    if (!out) return LC_ERR_NULL;
    // every check of lc_layout_copy over all tiles (a forced class, so any
    // overlap is refused), then one tile's logical modes
    Plan full, one;
    int st = make_plan(src, dst, w, n_tiles, LC_KERNEL_VEC_COPY, ptr, &full);
    if (st) return st;
    if ((st = make_plan(src, dst, w, 1, LC_KERNEL_VEC_COPY, PtrInfo{}, &one))) return st;
    LoopPlan lp;
    if ((st = check_loop(loop, one.total, &lp))) return st;
    lp.w = w;
    lp.n_tiles = n_tiles;
    lp.N = one.total;
    lp.logical = one.logical;
    lp.src_off = src->offset;
    lp.dst_off = dst->offset;
    int64_t cs, cd;
    if ((st = cosize(src, &cs)) || (st = cosize(dst, &cd))) return st;
    lp.sts = src->tile_stride ? src->tile_stride : cs;
    lp.dts = dst->tile_stride ? dst->tile_stride : cd;
    // widest vector of consecutive slots that is contiguous and aligned on
    // both sides in every tile ("copy -> gmem_smem" width rule)
    lp.vec = 1;
    const ModeList &lg = lp.logical;
    for (int bytes = 16; bytes >= 2 * w && lg.n > 0 && lp.N > 0; bytes /= 2) {
        const int v = bytes / w;
        const Mode &in = lg.m[lg.n - 1];
        bool ok = lp.inner_run % v == 0 && in.s == 1 && in.d == 1 && in.e % v == 0 &&
                  lp.src_off % v == 0 && lp.dst_off % v == 0;
        for (int i = 0; ok && i + 1 < lg.n; ++i) ok = lg.m[i].s % v == 0 && lg.m[i].d % v == 0;
        if (ok && n_tiles > 1) ok = lp.sts % v == 0 && lp.dts % v == 0;
        if (ok && ptr.check)
            ok = base_addr(ptr.src, lp.src_off, w) % uintptr_t(bytes) == 0 &&
                 base_addr(ptr.dst, lp.dst_off, w) % uintptr_t(bytes) == 0;
        if (ok) { lp.vec = v; break; }
    }
    // additive split: every suffix product of the loop modes and of the
    // logical modes (innermost first) lies on one divisibility chain
    if (lp.N > 0) {
        std::vector<int64_t> cuts;
        int64_t c = 1;
        for (int k = loop->rank - 1; k >= 0; --k) {
            if (loop->shape[k] == 1) continue;
            c *= loop->shape[k];
            cuts.push_back(c);
        }
        c = 1;
        for (int i = lg.n - 1; i >= 0; --i) {
            c *= lg.m[i].e;
            cuts.push_back(c);
        }
        std::sort(cuts.begin(), cuts.end());
        bool chain = true;
        int64_t prev = 1;
        for (int64_t x : cuts) {
            if (x % prev) { chain = false; break; }
            prev = x;
        }
        int64_t sspan = 1, dspan = 1;
        for (int i = 0; i < lg.n; ++i) {
            sspan += (lg.m[i].e - 1) * lg.m[i].s;
            dspan += (lg.m[i].e - 1) * lg.m[i].d;
        }
        lp.split = chain && sspan * w < (int64_t(1) << 31) && dspan * w < (int64_t(1) << 31);
    }
    *out = lp;
    return LC_OK;
}

}  // namespace lc

// ----------------------------------------------------------------------------
// host-only ABI entry points
// ----------------------------------------------------------------------------

extern "C" int lc_plan(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                       int32_t elem_bytes, int64_t n_tiles, int32_t kernel, lc_plan_info *out) {
    if (!out) return LC_ERR_NULL;
    lc::Plan p;
    lc::PtrInfo ptr;
    const int st = lc::make_plan(src_layout, dst_layout, elem_bytes, n_tiles, kernel, ptr, &p);
    if (st) return st;
    lc::fill_info(p, out);
    return LC_OK;
}

extern "C" int lc_choose_swizzle(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                                 int32_t elem_bytes, int32_t *k, int32_t *shift, int32_t *mask,
                                 int32_t *conflicts_read, int32_t *conflicts_write) {
    if (!src_layout || !dst_layout || !k || !shift || !mask || !conflicts_read || !conflicts_write)
        return LC_ERR_NULL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8 && elem_bytes != 16)
        return LC_ERR_ELEM_BYTES;
    lc::ModeList unit;
    const int st = lc::align_shards(src_layout, dst_layout, &unit);
    if (st) return st;
    int64_t total = 1;
    for (int i = 0; i < unit.n; ++i) total *= unit.m[i].e;
    if (total == 0 || total % 32) return LC_ERR_SHAPE;
    int kk, ss, rd, wd;
    const int bad = lc::choose_xor(unit, elem_bytes, &kk, &ss, &rd, &wd);
    *k = kk; *shift = ss; *mask = (1 << kk) - 1; *conflicts_read = rd; *conflicts_write = wd;
    return bad ? LC_ERR_NO_SWIZZLE : LC_OK;
}

extern "C" int lc_swizzle_conflicts(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                                    int32_t elem_bytes, int32_t k, int32_t shift,
                                    int32_t *conflicts_read, int32_t *conflicts_write) {
    if (!src_layout || !dst_layout || !conflicts_read || !conflicts_write) return LC_ERR_NULL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8 && elem_bytes != 16)
        return LC_ERR_ELEM_BYTES;
    if (k < 0 || k > 5 || shift < 0 || shift > 31) return LC_ERR_SHAPE;
    lc::ModeList unit;
    const int st = lc::align_shards(src_layout, dst_layout, &unit);
    if (st) return st;
    int64_t total = 1;
    for (int i = 0; i < unit.n; ++i) total *= unit.m[i].e;
    if (total == 0 || total % 32) return LC_ERR_SHAPE;
    int rd, wd;
    lc::phase_degrees(unit, elem_bytes, k, shift, &rd, &wd);
    *conflicts_read = rd;
    *conflicts_write = wd;
    return LC_OK;
}

namespace lc {
namespace {
// "copy -> gmem_smem", Algorithm step 1: the modes of a global / shared pair
// (s = global stride, d = shared stride) in the global side's canonical order,
// stride descending, neighbours contiguous on both sides merged.
int gmem_smem_modes(const lc_tile_layout *global_layout, const lc_tile_layout *shared_layout, ModeList *ml) {
    const int st = align_shards(global_layout, shared_layout, ml);
    if (st) return st;
    std::stable_sort(ml->m, ml->m + ml->n, [](const Mode &a, const Mode &b) { return a.s > b.s; });
    int n = 0;
    for (int i = 0; i < ml->n; ++i) {
        if (n && ml->m[n - 1].s == ml->m[i].s * ml->m[i].e && ml->m[n - 1].d == ml->m[i].d * ml->m[i].e) {
            ml->m[n - 1].e *= ml->m[i].e;
            ml->m[n - 1].s = ml->m[i].s;
            ml->m[n - 1].d = ml->m[i].d;
        } else {
            ml->m[n++] = ml->m[i];
        }
    }
    ml->n = n;
    return LC_OK;
}
}  // namespace
}  // namespace lc

extern "C" int lc_gmem_smem_plan(const lc_tile_layout *global_layout, const lc_tile_layout *shared_layout,
                                 int32_t elem_bytes, int32_t threads, const lc_smem_swizzle *swizzle,
                                 lc_gmem_smem *out) {
    if (!global_layout || !shared_layout || !out) return LC_ERR_NULL;
    if (!lc::valid_width(elem_bytes)) return LC_ERR_ELEM_BYTES;
    if (threads < 1 || threads > 1024) return LC_ERR_SHAPE;
    lc_smem_swizzle z{0, 0, 0};
    if (swizzle) z = *swizzle;
    if (z.bits < 0 || z.bits > 16 || z.chunk_log2 < 0 || z.chunk_log2 > 16 || z.row_log2 < 0 || z.row_log2 > 30)
        return LC_ERR_BAD_STRIDE;
    if (z.bits > 0 && (z.row_log2 < z.chunk_log2 + z.bits || (1 << z.chunk_log2) < elem_bytes))
        return LC_ERR_BAD_STRIDE;  // not one-to-one, or an element split across chunks
    for (const lc_tile_layout *l : {global_layout, shared_layout}) {
        if (l->rank < 1 || l->rank > LC_MAX_RANK) return LC_ERR_RANK;
        if (l->offset < 0) return LC_ERR_BAD_STRIDE;
        for (int k = 0; k < l->rank; ++k)
            if (l->shape[k] != 1 && l->stride[k] < 0) return LC_ERR_BAD_STRIDE;
    }
    lc::ModeList ml;
    int st = lc::gmem_smem_modes(global_layout, shared_layout, &ml);
    if (st) return st;
    int64_t total = 1;
    for (int i = 0; i < ml.n; ++i)
        if (!lc::mul_ok_ext(total, ml.m[i].e, &total) || total >= (int64_t(1) << 31)) return LC_ERR_SHAPE;
    std::memset(out, 0, sizeof(*out));
    out->n_modes = ml.n;
    for (int i = 0; i < ml.n; ++i) {
        out->extent[i] = ml.m[i].e;
        out->g_stride[i] = ml.m[i].s;
        out->s_stride[i] = ml.m[i].d;
        const lc::FastDiv fd = lc::make_fastdiv(static_cast<uint32_t>(ml.m[i].e ? ml.m[i].e : 1));
        out->div_m[i] = fd.m;
        out->div_s[i] = fd.s;
    }
    out->g_offset = global_layout->offset;
    out->s_offset = shared_layout->offset;
    out->elem_bytes = elem_bytes;
    out->threads = threads;
    out->total = total;
    out->swizzle = z;
    int v = 1;
    for (int bytes = 16; bytes > elem_bytes; bytes >>= 1) {
        if (z.bits > 0 && bytes > (1 << z.chunk_log2)) continue;  // one swizzle chunk at most
        const int c = bytes / elem_bytes;
        bool ok = ml.n > 0 && ml.m[ml.n - 1].s == 1 && ml.m[ml.n - 1].d == 1 && ml.m[ml.n - 1].e % c == 0 &&
                  out->g_offset % c == 0 && out->s_offset % c == 0;
        for (int i = 0; ok && i + 1 < ml.n; ++i) ok = ml.m[i].s % c == 0 && ml.m[i].d % c == 0;
        if (ok) { v = c; break; }
    }
    out->vec = v;
    const int64_t per_round = int64_t(threads) * v;
    out->outer = (total + per_round - 1) / per_round;
    out->guarded = total % per_round != 0;
    return LC_OK;
}

extern "C" int lc_gmem_smem_partition(const lc_tile_layout *global_layout,
                                      const lc_tile_layout *shared_layout, int32_t elem_bytes,
                                      int32_t threads, int32_t *vec, int64_t *outer) {
    if (!global_layout || !shared_layout || !vec || !outer) return LC_ERR_NULL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8 && elem_bytes != 16)
        return LC_ERR_ELEM_BYTES;
    if (threads < 1) return LC_ERR_SHAPE;
    lc::ModeList ml;
    int st = lc::gmem_smem_modes(global_layout, shared_layout, &ml);
    if (st) return st;
    int64_t total = 1;
    for (int i = 0; i < ml.n; ++i) total *= ml.m[i].e;
    if (total % threads) return LC_ERR_SHAPE;
    for (int bytes = 16; bytes >= elem_bytes; bytes >>= 1) {
        if (bytes % elem_bytes) continue;
        const int v = bytes / elem_bytes;
        bool ok = total % (int64_t(threads) * v) == 0;
        if (ok && v > 1) {
            ok = ml.n > 0 && ml.m[ml.n - 1].s == 1 && ml.m[ml.n - 1].d == 1 && ml.m[ml.n - 1].e % v == 0 &&
                 global_layout->offset % v == 0 && shared_layout->offset % v == 0;
            for (int i = 0; ok && i + 1 < ml.n; ++i) ok = ml.m[i].s % v == 0 && ml.m[i].d % v == 0;
        }
        if (ok) {
            *vec = v;
            *outer = total / (int64_t(threads) * v);
            return LC_OK;
        }
    }
    return LC_ERR_SHAPE;
}

extern "C" int lc_warp_unit_plan(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                                 int32_t elem_bytes, lc_warp_unit *out) {
    if (!src_layout || !dst_layout || !out) return LC_ERR_NULL;
    if (!lc::valid_width(elem_bytes)) return LC_ERR_ELEM_BYTES;
    for (int k = 0; k < src_layout->rank && k < LC_MAX_RANK; ++k)
        if (src_layout->stride[k] < 0) return LC_ERR_BAD_STRIDE;
    for (int k = 0; k < dst_layout->rank && k < LC_MAX_RANK; ++k)
        if (dst_layout->shape[k] != 1 && dst_layout->stride[k] <= 0) return LC_ERR_BAD_STRIDE;
    lc::ModeList unit;
    int st = lc::align_shards(src_layout, dst_layout, &unit);
    if (st) return st;
    if (unit.n > LC_MAX_RANK) return LC_ERR_SHAPE;
    int64_t total = 1;
    for (int i = 0; i < unit.n; ++i) total *= unit.m[i].e;
    if (total == 0 || total % 32 || total / 32 > LC_WARP_UNIT_MAX_P) return LC_ERR_SHAPE;
    // word offsets and byte spans stay in 31 bits on the device
    int64_t scos = 1, dcos = 1;
    for (int i = 0; i < unit.n; ++i) {
        scos += (unit.m[i].e - 1) * unit.m[i].s;
        dcos += (unit.m[i].e - 1) * unit.m[i].d;
    }
    if (scos * elem_bytes >= (int64_t(1) << 31) || dcos * elem_bytes >= (int64_t(1) << 31)) return LC_ERR_SHAPE;
    if ((st = lc::dst_injective(unit))) return st;
    lc_warp_unit u;
    std::memset(&u, 0, sizeof(u));
    u.n_modes = unit.n;
    for (int i = 0; i < unit.n; ++i) {
        u.extent[i] = static_cast<int32_t>(unit.m[i].e);
        u.src_stride[i] = static_cast<int32_t>(unit.m[i].s);
        u.dst_stride[i] = static_cast<int32_t>(unit.m[i].d);
    }
    u.P = static_cast<int32_t>(total / 32);
    int kk, ss, rd, wd;
    const int bad = lc::choose_xor(unit, elem_bytes, &kk, &ss, &rd, &wd);
    u.k = kk;
    u.shift = ss;
    u.mask = (1 << kk) - 1;
    u.conflicts_read = rd;
    u.conflicts_write = wd;
    u.src_cosize = static_cast<int32_t>(scos);
    u.dst_cosize = static_cast<int32_t>(dcos);
    *out = u;
    return bad ? LC_ERR_NO_SWIZZLE : LC_OK;
}

extern "C" int lc_loop_layout_default(int64_t n_elems, int32_t num_thread, int32_t vector_size,
                                      lc_loop_layout *out) {
    if (!out) return LC_ERR_NULL;
    if (n_elems < 0 || num_thread < 1 || vector_size < 1) return LC_ERR_SHAPE;
    const int64_t group = int64_t(num_thread) * vector_size;
    if (n_elems % group) return LC_ERR_SHAPE;
    std::memset(out, 0, sizeof(*out));
    out->rank = 3;
    out->shape[0] = n_elems / group;  // serial rounds
    out->slot_stride[0] = vector_size;
    out->shape[1] = num_thread;       // threads
    out->thread_stride[1] = 1;
    out->shape[2] = vector_size;      // points sharing a lane
    out->slot_stride[2] = 1;
    return LC_OK;
}

extern "C" int lc_loop_layout_info(const lc_loop_layout *loop, int64_t n_elems, int32_t *num_threads,
                                   int64_t *slots_per_thread) {
    lc::LoopPlan lp;
    const int st = lc::check_loop(loop, n_elems, &lp);
    if (st) return st;
    if (num_threads) *num_threads = static_cast<int32_t>(lp.T);
    if (slots_per_thread) *slots_per_thread = lp.L;
    return LC_OK;
}

extern "C" int lc_loop_plan(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                            int32_t elem_bytes, int64_t n_tiles, const lc_loop_layout *loop,
                            lc_loop_plan_info *out) {
    if (!out) return LC_ERR_NULL;
    lc::LoopPlan lp;
    lc::PtrInfo ptr;  // bases assumed aligned
    const int st = lc::make_loop_plan(src_layout, dst_layout, elem_bytes, n_tiles, loop, ptr, &lp);
    if (st) return st;
    out->num_threads = static_cast<int32_t>(lp.T);
    out->slots_per_thread = lp.L;
    out->points_per_tile = lp.N;
    out->vec = lp.vec;
    out->split = lp.split ? 1 : 0;
    return LC_OK;
}

extern "C" int lc_row_major_strides(int32_t rank, const int64_t *shape, int64_t *stride) {
    if (!shape || !stride) return LC_ERR_NULL;
    if (rank < 1 || rank > LC_MAX_RANK) return LC_ERR_RANK;
    int64_t acc = 1;
    for (int k = rank - 1; k >= 0; --k) {
        if (shape[k] < 0) return LC_ERR_SHAPE;
        stride[k] = acc;
        if (!lc::mul_ok_ext(acc, shape[k] > 1 ? shape[k] : 1, &acc)) return LC_ERR_OVERFLOW;
    }
    return LC_OK;
}

extern "C" int64_t lc_layout_footprint(const lc_tile_layout *l, int64_t n_tiles) {
    if (!l || l->rank < 1 || l->rank > LC_MAX_RANK || n_tiles < 0 || l->offset < 0 || l->tile_stride < 0) return -1;
    bool empty = n_tiles == 0;
    for (int k = 0; k < l->rank; ++k) {
        if (l->shape[k] < 0 || l->stride[k] < 0) return -1;
        empty = empty || l->shape[k] == 0;
    }
    if (empty) return l->offset;
    int64_t cos = 1, t;
    for (int k = 0; k < l->rank; ++k)
        if (!lc::mul_ok_ext(l->shape[k] - 1, l->stride[k], &t) || !lc::add_ok_ext(cos, t, &cos)) return -1;
    const int64_t ts = l->tile_stride ? l->tile_stride : cos;
    int64_t out;
    if (!lc::mul_ok_ext(n_tiles - 1, ts, &t) || !lc::add_ok_ext(t, cos, &out) || !lc::add_ok_ext(out, l->offset, &out))
        return -1;
    return out;
}
