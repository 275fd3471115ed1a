// CUDA C++ emission for a plan: three kernels, fully unrolled per path, CG non-zeros baked in
// as immediates ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
// abstract: static analysis at model compile time, sub-kernels whose operands live in
// registers, long arithmetic instruction streams).
//
//   uvu_fwd       receiver-stationary streaming forward: one thread per (receiver, channel,
//                 register group); the receiver's edges are scanned in CSR order and the output
//                 row is reduced in registers ("Receiver-streaming convolutions for channel-wise
//                 UVU tensor products", opening post, ownership paragraph).
//   uvu_bwd_edge  edges of a receiver, channels in parallel: dw stored directly, dY reduced over
//                 channels with warp shuffles and a fixed-order shared-memory sum, optional
//                 atomic dx scatter (same post, backward paragraph).
//   uvu_bwd_dx    sender-stationary dx over the transposed CSR, written once, no atomics
//                 (same page, reply on source- vs destination-stationary convolutions).
//
// Per-edge arithmetic of one path p = (l1, l2, l3) for one channel, with q[a,b] = x[a] y[b]:
//   forward   t[m3] = sum_nz c q[m1,m2];            acc[m3] += w_p t[m3]
//   dw        dw_p  = sum_m3 g[m3] t[m3]
//   dY, dx    h[m1,m2] += sum_nz c (w_p g[m3]);     dY[m2] += sum_m1 x[m1] h;  dx[m1] += sum_m2 y[m2] h
// where h is accumulated over all paths sharing (l1, l2) before it is contracted.
// Paths whose CG is a signed permutation with a scalar operand (l1 = 0 or l2 = 0) skip the
// products: acc[m3] += (w_p x0) (+-y[m2]).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <map>
#include <set>
#include <sstream>
#include <string>
#include <vector>

#include "plan.h"

namespace uvu {
namespace {

struct Src {
    std::ostringstream o;
    int ind = 0;
    Src& operator()(const std::string& s) {
        for (int i = 0; i < ind; ++i) o << "  ";
        o << s << "\n";
        return *this;
    }
};

std::string fmt(const char* f, ...) __attribute__((format(printf, 1, 2)));
std::string fmt(const char* f, ...) {
    va_list ap, ap2;
    va_start(ap, f);
    va_copy(ap2, ap);
    const int n = vsnprintf(nullptr, 0, f, ap);
    va_end(ap);
    std::string out(n > 0 ? size_t(n) : 0, '\0');
    if (n > 0) vsnprintf(&out[0], size_t(n) + 1, f, ap2);  // writes the terminator into the spare byte
    va_end(ap2);
    return out;
}

struct Gen {
    Plan* P;
    bool f64;
    std::string T;

    std::string lit(double c) const {
        char b[64];
        if (f64) {
            snprintf(b, sizeof b, "%.17e", c);
            return b;
        }
        snprintf(b, sizeof b, "%.9ef", double(float(c)));
        return b;
    }
    static bool is_one(double c) { return std::abs(std::abs(c) - 1.0) < 1e-14; }

    // A path whose CG maps each m3 to exactly one (m1, m2) with coefficient +-1 and one operand
    // of width 1: the identity couplings (0, l, l) and (l, 0, l).
    // Set while emitting the double-backward kernels, whose operands are sums of products and
    // therefore always take the generic path.
    mutable bool no_identity = false;
    // dw of a path: stored per edge (dwe[p * U]) or, for weights shared by a whole batch,
    // accumulated in the thread's registers (dwa_p) over the samples it processes
    mutable bool dw_accum = false;
    // Set while emitting the plain edge kernel with a wide output row: the x (x) y products of an
    // (x irrep, SH irrep) pair are formed inside that pair's block, just before its paths use
    // them, instead of all at once before the paths (fewer values live at a time).
    mutable bool local_products = false;
    // guard_dw: the store is skipped when dw is NULL (the one-pass emission computes dw with the
    // rest of the path instead of in a block of its own under that condition)
    mutable bool guard_dw = false;
    std::string dw_store(int pi, const std::string& v) const {
        if (dw_accum) return fmt("dwa_%d += %s;", pi, v.c_str());
        return fmt("%sdwe[%d * UVU_U] = %s;", guard_dw ? "if (dw) " : "", pi, v.c_str());
    }

    bool is_identity(const PathInfo& p) const {
        if (no_identity) return false;
        if (p.l1 != 0 && p.l2 != 0) return false;
        std::vector<int> cnt(2 * p.l3 + 1, 0);
        for (const Nz& z : p.nz) {
            if (!is_one(z.c)) return false;
            cnt[z.m3]++;
        }
        for (int c : cnt)
            if (c != 1) return false;
        return true;
    }

    // Column scales of the d_out row: for each output index k = ooff + m3 of a general path, the
    // magnitude shared by most CG entries of that (path, m3) column (1 for identity paths).  A
    // kernel that keeps a receiver's d_out row in registers for all of its edges loads s_k g_k
    // once per receiver and uses C / s_k, so the column's most common coefficient becomes +-1:
    // the t row of dw starts without a multiply, and so do the h entries first reached through
    // such a coefficient.  Set only while emitting such a kernel.
    mutable const std::vector<double>* colscale = nullptr;
    // Set while emitting an fp32 edge kernel whose dY and dx contractions use paired FMAs (h
    // entries of adjacent SH components as one register pair; xb_a = {x_a, x_a}; dxq_a the even
    // and odd partial sums of dx_a).
    mutable bool pair_contract = false;
    // with pair_contract: only dY's contraction paired, {x_a, x_a} formed at each use (no
    // per-edge pair registers), dx's contraction scalar (the staged-row kernels' register budget)
    mutable bool pair_dy_only = false;
    // Identity paths (0,l,l) and (l,0,l) in the plain edge kernels: zi_p = sum of +-g x (or g y)
    // over the path's pairs serves dw (zi_p times the width-1 operand), dY (l2 = 0: w zi_p) or dx
    // (l1 = 0: w zi_p), and the other gradient takes (w times the width-1 operand) g directly:
    // no h entries, no a = w g products.  zi_ready: paths whose zi_p is already in scope.
    mutable bool id_fold = false;
    mutable std::set<int> zi_ready;
    static bool id_fold_enabled() {
        const char* e = std::getenv("UVU_ID_FOLD");
        return !(e && std::atoi(e) == 0);
    }
    template <class GV>
    void emit_identity_z(Src& S, int pi, GV gval, const char* xname = "xv", const char* yname = "yv") const {
        const PathInfo& p = P->paths[pi];
        const bool scal_x = (p.l1 == 0);
        bool first = true;
        for (const Nz& z : p.nz) {
            const std::string other = scal_x ? fmt("%s_%d", yname, p.yoff + z.m2) : fmt("%s_%d", xname, p.xoff + z.m1);
            const std::string gv = gval(p.ooff + z.m3);
            if (first)
                S(fmt("%s zi_%d = %s%s * %s;", T.c_str(), pi, z.c < 0 ? "-" : "", gv.c_str(), other.c_str()));
            else
                S(fmt("zi_%d = fma(%s%s, %s, zi_%d);", pi, z.c < 0 ? "-" : "", gv.c_str(), other.c_str(), pi));
            first = false;
        }
    }
    double cs(int k) const { return colscale ? (*colscale)[k] : 1.0; }
    std::vector<double> column_scales() const {
        std::vector<double> s(P->Do, 1.0);
        for (const PathInfo& p : P->paths) {
            if (is_identity(p)) continue;
            for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3) {
                std::vector<std::pair<double, int>> mags;  // (magnitude, count) in first-seen order
                for (const Nz& z : p.nz) {
                    if (z.m3 != m3) continue;
                    const double a = std::abs(z.c);
                    bool found = false;
                    for (auto& mc : mags)
                        if (std::abs(mc.first - a) <= 1e-13 * a) { mc.second++; found = true; break; }
                    if (!found) mags.push_back({a, 1});
                }
                int best = -1;
                for (size_t i = 0; i < mags.size(); ++i)
                    if (best < 0 || mags[i].second > mags[size_t(best)].second) best = int(i);
                if (best >= 0) s[size_t(p.ooff + m3)] = mags[size_t(best)].first;
            }
        }
        return s;
    }
    // UVU_COL_SCALE=0 (a tuning switch) emits the unscaled form.
    // The plain edge kernel with one-edge stages writes dw and the per-edge dx partials into the
    // stage it read w and x from (same shapes: [P][U] and [U][D_x]) and one thread moves them to
    // global memory with two bulk copies per stage: no per-thread global stores (whose register
    // operands the warps otherwise wait on) and full-line writes.  Measured: wide (U = 256) VJP
    // 5.89 -> 5.33 ms, MACE-large and fp64 unchanged; MACE-medium (two-edge stages, released
    // per warp otherwise) 0.777 -> 0.818 ms, so two-edge stages keep the per-thread stores.
    // UVU_EDGE_BULK_OUT=0 (a tuning switch) keeps them everywhere.
    static bool edge_bulk_out_enabled() {
        const char* e = std::getenv("UVU_EDGE_BULK_OUT");
        return !(e && std::atoi(e) == 0);
    }
    mutable bool obulk = false;
    // Set while emitting the one-pass edge kernel that reads d_out from the staged block: each
    // path's d_out values are read once at the top of its block, two at a time (8- or 16-byte
    // shared-memory loads at even columns, so only for an even D_out, where every row starts
    // at an even element offset), into gq_k.  UVU_GSM_VEC=0 (a tuning switch) reads each value
    // where it is used.
    mutable bool gsm_vec = false;
    static bool gsm_vec_enabled() {
        const char* e = std::getenv("UVU_GSM_VEC");
        return !(e && std::atoi(e) == 0);
    }
    // Words per warp of the dY tile: 32 rows of 16, rows 16..31 shifted by 16 words so that the
    // two half-warps' column reads fall in opposite bank halves.
    static constexpr int kDytWords = 528;
    // UVU_DY_SMEM=0 (a tuning switch) keeps the shuffle transpose-reduce for dY.
    static bool dy_smem_enabled() {
        const char* e = std::getenv("UVU_DY_SMEM");
        return !(e && std::atoi(e) == 0);
    }
    static bool pair_contract_enabled() {
        const char* e = std::getenv("UVU_PAIR_CONTRACT");
        return !(e && std::atoi(e) == 0);
    }
    static bool col_scale_enabled() {
        const char* e = std::getenv("UVU_COL_SCALE");
        return !(e && std::atoi(e) == 0);
    }
    // d_out value k as loaded: scaled by its column scale when one is in force
    std::string gload(int k, const std::string& v) const {
        const double sk = cs(k);
        return sk == 1.0 ? v : fmt("%s * %s", lit(sk).c_str(), v.c_str());
    }

    std::set<int> x_needed(const std::vector<int>& paths) const {
        std::set<int> s;
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            for (int m = 0; m < 2 * p.l1 + 1; ++m) s.insert(p.xoff + m);
        }
        return s;
    }
    std::set<int> y_needed(const std::vector<int>& paths) const {
        std::set<int> s;
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            for (int m = 0; m < 2 * p.l2 + 1; ++m) s.insert(p.yoff + m);
        }
        return s;
    }

    // Emit loads "T pre_k = base[k]" for k in `need`, with 16-byte vector loads when the row
    // stride keeps every row 16-byte aligned.
    void emit_row_loads(Src& S, const std::string& pre, const std::string& base, int width,
                        const std::set<int>& need, bool global = true) const {
        const int esz = f64 ? 8 : 4;
        const int V = 16 / esz;
        if ((width * esz) % 16 == 0) {
            const std::string VT = f64 ? "double2" : "float4";
            std::set<int> chunks;
            for (int k : need) chunks.insert(k / V);
            S(fmt("const %s* %s_v = reinterpret_cast<const %s*>(%s);", VT.c_str(), pre.c_str(),
                  VT.c_str(), base.c_str()));
            for (int c : chunks) {
                if (global)
                    S(fmt("const %s %s_c%d = __ldg(%s_v + %d);", VT.c_str(), pre.c_str(), c, pre.c_str(), c));
                else
                    S(fmt("const %s %s_c%d = %s_v[%d];", VT.c_str(), pre.c_str(), c, pre.c_str(), c));
                static const char* comp[4] = {"x", "y", "z", "w"};
                for (int i = 0; i < V; ++i) {
                    const int k = c * V + i;
                    if (need.count(k))
                        S(fmt("const %s %s_%d = %s_c%d.%s;", T.c_str(), pre.c_str(), k, pre.c_str(), c, comp[i]));
                }
            }
        } else {
            for (int k : need) {
                if (global)
                    S(fmt("const %s %s_%d = __ldg(%s + %d);", T.c_str(), pre.c_str(), k, base.c_str(), k));
                else
                    S(fmt("const %s %s_%d = (%s)[%d];", T.c_str(), pre.c_str(), k, base.c_str(), k));
            }
        }
    }

    // fp32 products of an x value with two y values at even/odd index pairs use one paired
    // multiply (mul.rn.f32x2, each half rounded as a scalar multiply, so the results are the same
    // bits).  Measured on MACE-medium: forward 0.356 -> 0.339 ms, edge kernel 0.862 -> 0.820 ms
    // (fewer issue slots in issue-bound kernels); MACE-large unchanged.  UVU_PACK_PRODUCTS=0 (a
    // tuning switch) emits scalar multiplies.
    bool pack_products() const {
        return !f64 && !(std::getenv("UVU_PACK_PRODUCTS") && std::atoi(std::getenv("UVU_PACK_PRODUCTS")) == 0);
    }
    // Device helpers of the paired fp32 products (emitted when they are used).
    void emit_pair_helpers(Src& S) const {
        if (!pack_products()) return;
        S("__device__ __forceinline__ unsigned long long uvu_f2pack(float a, float b) {");
        S("  unsigned long long r; asm(\"mov.b64 %0, {%1, %2};\" : \"=l\"(r) : \"f\"(a), \"f\"(b)); return r; }");
        S("__device__ __forceinline__ void uvu_f2unpack(unsigned long long v, float& a, float& b) {");
        S("  asm(\"mov.b64 {%0, %1}, %2;\" : \"=f\"(a), \"=f\"(b) : \"l\"(v)); }");
        S("__device__ __forceinline__ unsigned long long uvu_f2mul(unsigned long long a, unsigned long long b) {");
        S("  unsigned long long d; asm(\"mul.rn.f32x2 %0, %1, %2;\" : \"=l\"(d) : \"l\"(a), \"l\"(b)); return d; }");
        S("__device__ __forceinline__ unsigned long long uvu_f2fma(unsigned long long a, unsigned long long b, unsigned long long c) {");
        S("  unsigned long long d; asm(\"fma.rn.f32x2 %0, %1, %2, %3;\" : \"=l\"(d) : \"l\"(a), \"l\"(b), \"l\"(c)); return d; }");
    }

    // Products q_a_b = xv_a * yv_b used by the non-identity paths in `paths`.
    void emit_products(Src& S, const std::vector<int>& paths) const {
        std::set<std::pair<int, int>> q;
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            if (is_identity(p)) continue;
            for (const Nz& z : p.nz) q.insert({p.xoff + z.m1, p.yoff + z.m2});
        }
        if (!pack_products()) {
            for (auto& ab : q)
                S(fmt("const %s q_%d_%d = xv_%d * yv_%d;", T.c_str(), ab.first, ab.second, ab.first, ab.second));
            return;
        }
        std::map<int, std::set<int>> byx;
        for (auto& ab : q) byx[ab.first].insert(ab.second);
        for (auto& kv : byx) {
            const int a = kv.first;
            const std::set<int>& bs = kv.second;
            std::vector<int> pairs, singles;
            for (int b : bs) {
                if (b % 2 == 0 && bs.count(b + 1)) pairs.push_back(b);
                else if (b % 2 == 1 && bs.count(b - 1)) continue;
                else singles.push_back(b);
            }
            if (!pairs.empty()) S(fmt("const unsigned long long xx_%d = uvu_f2pack(xv_%d, xv_%d);", a, a, a));
            for (int b : pairs)
                S(fmt("float q_%d_%d, q_%d_%d; uvu_f2unpack(uvu_f2mul(xx_%d, uvu_f2pack(yv_%d, yv_%d)), q_%d_%d, q_%d_%d);", a, b, a,
                      b + 1, a, b, b + 1, a, b, a, b + 1));
            for (int b : singles) S(fmt("const float q_%d_%d = xv_%d * yv_%d;", a, b, a, b));
        }
    }

    // <tpre>_<p>_<m3> = sum_nz c <qpre>_<a>_<b>   (general paths only)
    void emit_t(Src& S, int pi, const char* qpre = "q", const char* tpre = "t") const {
        const PathInfo& p = P->paths[pi];
        for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3) {
            std::vector<std::pair<double, std::string>> terms;
            for (const Nz& z : p.nz) {
                if (z.m3 != m3) continue;
                terms.push_back({z.c / cs(p.ooff + m3), fmt("%s_%d_%d", qpre, p.xoff + z.m1, p.yoff + z.m2)});
            }
            if (colscale)  // a +-1 term first: the row then starts without a multiply
                for (size_t i = 1; i < terms.size(); ++i)
                    if (!is_one(terms[0].first) && is_one(terms[i].first)) std::swap(terms[0], terms[i]);
            bool first = true;
            for (const auto& tm : terms) {
                const double c = tm.first;
                const std::string& q = tm.second;
                if (first) {
                    if (is_one(c))
                        S(fmt("%s %s_%d_%d = %s%s;", T.c_str(), tpre, pi, m3, c < 0 ? "-" : "", q.c_str()));
                    else
                        S(fmt("%s %s_%d_%d = %s * %s;", T.c_str(), tpre, pi, m3, lit(c).c_str(), q.c_str()));
                    first = false;
                } else if (colscale && is_one(c)) {
                    S(fmt("%s_%d_%d %s= %s;", tpre, pi, m3, c < 0 ? "-" : "+", q.c_str()));
                } else {
                    S(fmt("%s_%d_%d = fma(%s, %s, %s_%d_%d);", tpre, pi, m3, lit(c).c_str(), q.c_str(), tpre, pi, m3));
                }
            }
            if (first) S(fmt("const %s %s_%d_%d = 0;", T.c_str(), tpre, pi, m3));
        }
    }

    // ------------------------------------------------------------------ forward
    // acc_* += contribution of one edge, from xv_*, yv_*, wv_* already in registers.
    // Sender-stationary forward (source-stationary convolution): one thread per (sender, register
    // group, channel) keeps its x row in registers, walks the sender's out-edges over the
    // transposed CSR and adds each edge's contribution to out[recv] with reduction atomics (out
    // zeroed first).  The alternative to the receiver-stationary forward when x rows are wider
    // than out rows ("Receiver-streaming convolutions ...", replies: source- and destination-
    // stationary convolutions, the one that moves less data chosen at init time).
    void emit_fwd_sender_group(Src& S, int g) const {
        const std::vector<int>& paths = P->groups[g];
        const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
        std::vector<int> outs;
        for (int pi : paths)
            for (int m = 0; m < 2 * P->paths[pi].l3 + 1; ++m) outs.push_back(P->paths[pi].ooff + m);
        S(fmt("__device__ __forceinline__ void fsend_group%d(int k0, int k1, int u, const int* __restrict__ seid,", g));
        S(fmt("    const int* __restrict__ srecv, const %s* __restrict__ xrow, const %s* __restrict__ Y,", T.c_str(), T.c_str()));
        S(fmt("    const %s* __restrict__ w, %s* __restrict__ out) {", T.c_str(), T.c_str()));
        S.ind++;
        emit_row_loads(S, "xv", "xrow", P->Dx, xn);
        S("#pragma unroll 1");
        S("for (int k = k0; k < k1; ++k) {");
        S.ind++;
        S("const int e = __ldg(seid + k), r = __ldg(srecv + k);");
        emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        S("const " + T + "* __restrict__ we = w + (size_t)e * (UVU_P * UVU_U) + u;");
        for (int pi : paths) S(fmt("const %s wv_%d = __ldg(we + %d * UVU_U);", T.c_str(), pi, pi));
        for (int k : outs) S(fmt("%s acc_%d = 0;", T.c_str(), k));
        emit_fwd_edge(S, paths);
        S(T + "* __restrict__ orow = out + ((size_t)r * UVU_U + u) * UVU_DO;");
        for (int k : outs) S(fmt("atomicAdd(orow + %d, acc_%d);", k, k));
        S.ind--;
        S("}");
        S.ind--;
        S("}");
    }
    void emit_fwd_sender_kernel(Src& S) const {
        const int NG = int(P->groups.size());
        for (int g = 0; g < NG; ++g) emit_fwd_sender_group(S, g);
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_FS_TPB) uvu_fwd_sender(long long N, const int* __restrict__ soff,"));
        S(fmt("    const int* __restrict__ seid, const int* __restrict__ srecv, const %s* __restrict__ x,", T.c_str()));
        S(fmt("    const %s* __restrict__ Y, const %s* __restrict__ w, %s* __restrict__ out) {", T.c_str(), T.c_str(), T.c_str()));
        S("  const int u = threadIdx.x % UVU_UP;");
        S("  const int g = (threadIdx.x / UVU_UP) % UVU_G;");
        S("  const long long sn = (long long)blockIdx.x * UVU_FS_SPB + threadIdx.x / (UVU_UP * UVU_G);");
        S("  if (sn >= N || u >= UVU_U) return;");
        S("  const int k0 = __ldg(soff + sn), k1 = __ldg(soff + sn + 1);");
        S(fmt("  const %s* xrow = x + ((size_t)sn * UVU_U + u) * UVU_DX;", T.c_str()));
        for (int g = 0; g < NG; ++g)
            S(fmt("  %sif (g == %d) fsend_group%d(k0, k1, u, seid, srecv, xrow, Y, w, out);", g ? "else " : "", g, g));
        S("}");
    }

    void emit_fwd_edge(Src& S, const std::vector<int>& paths) const {
        emit_products(S, paths);
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            S(fmt("// path %d: (%d,%d,%d)", pi, p.l1, p.l2, p.l3));
            if (is_identity(p)) {
                const bool scal_x = (p.l1 == 0);
                S(fmt("{ const %s sw = wv_%d * %s;", T.c_str(), pi,
                      scal_x ? fmt("xv_%d", p.xoff).c_str() : fmt("yv_%d", p.yoff).c_str()));
                for (const Nz& z : p.nz) {
                    const std::string other = scal_x ? fmt("yv_%d", p.yoff + z.m2) : fmt("xv_%d", p.xoff + z.m1);
                    S(fmt("  acc_%d = fma(%ssw, %s, acc_%d);", p.ooff + z.m3, z.c < 0 ? "-" : "", other.c_str(), p.ooff + z.m3));
                }
                S("}");
            } else {
                S("{");
                S.ind++;
                emit_t(S, pi);
                for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3)
                    S(fmt("acc_%d = fma(wv_%d, t_%d_%d, acc_%d);", p.ooff + m3, pi, pi, m3, p.ooff + m3));
                S.ind--;
                S("}");
            }
        }
    }

    void emit_fwd_group(Src& S, int g) const {
        const std::vector<int>& paths = P->groups[g];
        S(fmt("__device__ __forceinline__ void fwd_group%d(int e0, int e1, int u, const int* __restrict__ src,", g));
        S(fmt("    const %s* __restrict__ x, const %s* __restrict__ Y, const %s* __restrict__ w, %s* __restrict__ orow) {",
              T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        S.ind++;
        std::vector<int> outs;
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            for (int m = 0; m < 2 * p.l3 + 1; ++m) outs.push_back(p.ooff + m);
        }
        for (int k : outs) S(fmt("%s acc_%d = 0;", T.c_str(), k));
        const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
        S("#pragma unroll 1");
        S("for (int e = e0; e < e1; ++e) {");
        S.ind++;
        S("const int s = __ldg(src + e);");
        emit_row_loads(S, "xv", fmt("x + ((size_t)s * UVU_U + u) * UVU_DX"), P->Dx, xn);
        emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        S("const " + T + "* __restrict__ we = w + (size_t)e * (UVU_P * UVU_U) + u;");
        for (int pi : paths) S(fmt("const %s wv_%d = __ldg(we + %d * UVU_U);", T.c_str(), pi, pi));
        emit_fwd_edge(S, paths);
        S.ind--;
        S("}");
        for (int k : outs) S(fmt("orow[%d] = acc_%d;", k, k));
        S.ind--;
        S("}");
    }

    // ------------------------------------------------------------------ per-pair backward core
    // Emits, for the paths of `paths` grouped by (ix, iy): optional dw stores, then the h
    // accumulation and its contraction into dyp_* (if want_dy) and dxp_* (if want_dx).
    // gval(k) names the d_out value of output index k.
    template <class GV>
    void emit_bwd_pairs(Src& S, const std::vector<int>& paths, bool want_dw, bool want_dy,
                        bool want_dx, GV gval, const char* xname = "xv", const char* yname = "yv",
                        const char* wname = "wv") const {
        std::map<std::pair<int, int>, std::vector<int>> pairs;
        for (int pi : paths) pairs[{P->paths[pi].ix, P->paths[pi].iy}].push_back(pi);
        for (auto& kv : pairs) {
            const std::vector<int>& pp = kv.second;
            const PathInfo& p0 = P->paths[pp[0]];
            const int d1 = 2 * p0.l1 + 1, d2 = 2 * p0.l2 + 1;
            S("{");
            S.ind++;
            if (local_products && want_dw) emit_products(S, pp);
            std::set<std::pair<int, int>> hdef;
            for (int pi : pp) {
                const PathInfo& p = P->paths[pi];
                S(fmt("// path %d: (%d,%d,%d)", pi, p.l1, p.l2, p.l3));
                if (gsm_vec) {
                    const int d3 = 2 * p.l3 + 1;
                    const std::string T2 = f64 ? "double2" : "float2";
                    for (int m3 = 0; m3 < d3; ++m3) {
                        const int k = p.ooff + m3;
                        if (k % 2 == 0 && m3 + 1 < d3) {
                            S(fmt("const %s gq2_%d = *reinterpret_cast<const %s*>(grow + %d);", T2.c_str(), k, T2.c_str(), k));
                            S(fmt("const %s gq_%d = gq2_%d.x, gq_%d = gq2_%d.y;", T.c_str(), k, k, k + 1, k));
                            ++m3;
                        } else {
                            S(fmt("const %s gq_%d = grow[%d];", T.c_str(), k, k));
                        }
                    }
                }
                if (id_fold && is_identity(p)) {
                    const bool scal_x = (p.l1 == 0);
                    const std::string x0 = fmt("%s_%d", xname, p.xoff), y0 = fmt("%s_%d", yname, p.yoff);
                    if (!zi_ready.count(pi)) emit_identity_z(S, pi, gval, xname, yname);
                    if (want_dw) S(dw_store(pi, fmt("zi_%d * %s", pi, scal_x ? x0.c_str() : y0.c_str())));
                    if (scal_x) {  // (0, l, l): dx_0 += w zi; dY_m2 += c (x_0 w) g_m3
                        if (want_dx) S(fmt("dxp_%d = fma(%s_%d, zi_%d, dxp_%d);", p.xoff, wname, pi, pi, p.xoff));
                        if (want_dy) {
                            S(fmt("const %s xw_%d = %s * %s_%d;", T.c_str(), pi, x0.c_str(), wname, pi));
                            for (const Nz& z : p.nz)
                                S(fmt("dyp_%d = fma(%sxw_%d, %s, dyp_%d);", p.yoff + z.m2, z.c < 0 ? "-" : "", pi,
                                      gval(p.ooff + z.m3).c_str(), p.yoff + z.m2));
                        }
                    } else {  // (l, 0, l): dY_0 += w zi; dx_m1 += c (y_0 w) g_m3
                        if (want_dy) S(fmt("dyp_%d = fma(%s_%d, zi_%d, dyp_%d);", p.yoff, wname, pi, pi, p.yoff));
                        if (want_dx) {
                            S(fmt("const %s yw_%d = %s * %s_%d;", T.c_str(), pi, y0.c_str(), wname, pi));
                            for (const Nz& z : p.nz)
                                S(fmt("dxp_%d = fma(%syw_%d, %s, dxp_%d);", p.xoff + z.m1, z.c < 0 ? "-" : "", pi,
                                      gval(p.ooff + z.m3).c_str(), p.xoff + z.m1));
                        }
                    }
                    continue;
                }
                if (want_dw) {
                    if (is_identity(p)) {
                        const bool scal_x = (p.l1 == 0);
                        bool first = true;
                        for (const Nz& z : p.nz) {
                            const std::string other = scal_x ? fmt("yv_%d", p.yoff + z.m2) : fmt("xv_%d", p.xoff + z.m1);
                            const std::string gv = gval(p.ooff + z.m3);
                            if (first) {
                                S(fmt("%s z_%d = %s%s * %s;", T.c_str(), pi, z.c < 0 ? "-" : "", gv.c_str(), other.c_str()));
                                first = false;
                            } else {
                                S(fmt("z_%d = fma(%s%s, %s, z_%d);", pi, z.c < 0 ? "-" : "", gv.c_str(), other.c_str(), pi));
                            }
                        }
                        S(dw_store(pi, fmt("z_%d * %s", pi, scal_x ? fmt("xv_%d", p.xoff).c_str() : fmt("yv_%d", p.yoff).c_str())));
                    } else {
                        S("{");
                        S.ind++;
                        emit_t(S, pi);
                        for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3) {
                            if (m3 == 0)
                                S(fmt("%s z = %s * t_%d_0;", T.c_str(), gval(p.ooff).c_str(), pi));
                            else
                                S(fmt("z = fma(%s, t_%d_%d, z);", gval(p.ooff + m3).c_str(), pi, m3));
                        }
                        S(dw_store(pi, "z"));
                        S.ind--;
                        S("}");
                    }
                }
                if ((want_dy || want_dx) && colscale) {
                    for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3)
                        S(fmt("const %s a_%d_%d = %s_%d * %s;", T.c_str(), pi, m3, wname, pi, gval(p.ooff + m3).c_str()));
                    // this path's contributions per h entry; an entry not yet defined takes a +-1
                    // contribution as its definition when it has one
                    std::map<std::pair<int, int>, std::vector<std::pair<double, std::string>>> by;
                    for (const Nz& z : p.nz)
                        by[{p.xoff + z.m1, p.yoff + z.m2}].push_back({z.c / cs(p.ooff + z.m3), fmt("a_%d_%d", pi, z.m3)});
                    for (auto& kv : by) {
                        const int a = kv.first.first, b = kv.first.second;
                        auto& L = kv.second;
                        if (!hdef.count({a, b})) {
                            for (size_t i = 1; i < L.size(); ++i)
                                if (!is_one(L[0].first) && is_one(L[i].first)) std::swap(L[0], L[i]);
                        }
                        for (size_t i = 0; i < L.size(); ++i) {
                            const double c = L[i].first;
                            const std::string& av = L[i].second;
                            if (!hdef.count({a, b})) {
                                hdef.insert({a, b});
                                if (is_one(c))
                                    S(fmt("%s h_%d_%d = %s%s;", T.c_str(), a, b, c < 0 ? "-" : "", av.c_str()));
                                else
                                    S(fmt("%s h_%d_%d = %s * %s;", T.c_str(), a, b, lit(c).c_str(), av.c_str()));
                            } else if (is_one(c)) {
                                S(fmt("h_%d_%d %s= %s;", a, b, c < 0 ? "-" : "+", av.c_str()));
                            } else {
                                S(fmt("h_%d_%d = fma(%s, %s, h_%d_%d);", a, b, lit(c).c_str(), av.c_str(), a, b));
                            }
                        }
                    }
                } else if (want_dy || want_dx) {
                    for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3)
                        S(fmt("const %s a_%d_%d = %s_%d * %s;", T.c_str(), pi, m3, wname, pi, gval(p.ooff + m3).c_str()));
                    for (const Nz& z : p.nz) {
                        const int a = p.xoff + z.m1, b = p.yoff + z.m2;
                        const std::string av = fmt("a_%d_%d", pi, z.m3);
                        if (!hdef.count({a, b})) {
                            hdef.insert({a, b});
                            if (is_one(z.c))
                                S(fmt("%s h_%d_%d = %s%s;", T.c_str(), a, b, z.c < 0 ? "-" : "", av.c_str()));
                            else
                                S(fmt("%s h_%d_%d = %s * %s;", T.c_str(), a, b, lit(z.c).c_str(), av.c_str()));
                        } else {
                            if (is_one(z.c))
                                S(fmt("h_%d_%d %s= %s;", a, b, z.c < 0 ? "-" : "+", av.c_str()));
                            else
                                S(fmt("h_%d_%d = fma(%s, %s, h_%d_%d);", a, b, lit(z.c).c_str(), av.c_str(), a, b));
                        }
                    }
                }
            }
            if (pair_contract && (want_dy || want_dx)) {
                // h entries (a, b), (a, b+1) with b even as one register pair: dY's pair (b, b+1)
                // and dx's even/odd partial sums each take one paired FMA per pair
                for (int m1 = 0; m1 < d1; ++m1) {
                    const int a = p0.xoff + m1;
                    for (int m2 = 0; m2 < d2; ++m2) {
                        const int b = p0.yoff + m2;
                        if (!hdef.count({a, b})) continue;
                        const bool pr = b % 2 == 0 && m2 + 1 < d2 && hdef.count({a, b + 1});
                        const bool second = b % 2 == 1 && m2 > 0 && hdef.count({a, b - 1});
                        if (second) continue;
                        if (pr && pair_dy_only) {
                            if (want_dy)
                                S(fmt("{ unsigned long long d = uvu_f2pack(dyp_%d, dyp_%d); d = uvu_f2fma(uvu_f2pack(%s_%d, %s_%d), "
                                      "uvu_f2pack(h_%d_%d, h_%d_%d), d); uvu_f2unpack(d, dyp_%d, dyp_%d); }",
                                      b, b + 1, xname, a, xname, a, a, b, a, b + 1, b, b + 1));
                            if (want_dx) {
                                S(fmt("dxp_%d = fma(%s_%d, h_%d_%d, dxp_%d);", a, yname, b, a, b, a));
                                S(fmt("dxp_%d = fma(%s_%d, h_%d_%d, dxp_%d);", a, yname, b + 1, a, b + 1, a));
                            }
                        } else if (pr) {
                            S(fmt("{ const unsigned long long hp = uvu_f2pack(h_%d_%d, h_%d_%d);", a, b, a, b + 1));
                            if (want_dy)
                                S(fmt("  { unsigned long long d = uvu_f2pack(dyp_%d, dyp_%d); d = uvu_f2fma(xb_%d, hp, d); "
                                      "uvu_f2unpack(d, dyp_%d, dyp_%d); }", b, b + 1, a, b, b + 1));
                            if (want_dx) S(fmt("  dxq_%d = uvu_f2fma(uvu_f2pack(%s_%d, %s_%d), hp, dxq_%d);", a, yname, b, yname, b + 1, a));
                            S("}");
                        } else {
                            if (want_dy) S(fmt("dyp_%d = fma(%s_%d, h_%d_%d, dyp_%d);", b, xname, a, a, b, b));
                            if (want_dx) S(fmt("dxp_%d = fma(%s_%d, h_%d_%d, dxp_%d);", a, yname, b, a, b, a));
                        }
                    }
                }
            }
            if (want_dy && !pair_contract) {
                for (int m2 = 0; m2 < d2; ++m2) {
                    const int b = p0.yoff + m2;
                    for (int m1 = 0; m1 < d1; ++m1) {
                        const int a = p0.xoff + m1;
                        if (hdef.count({a, b})) S(fmt("dyp_%d = fma(%s_%d, h_%d_%d, dyp_%d);", b, xname, a, a, b, b));
                    }
                }
            }
            if (want_dx && !pair_contract) {
                for (int m1 = 0; m1 < d1; ++m1) {
                    const int a = p0.xoff + m1;
                    for (int m2 = 0; m2 < d2; ++m2) {
                        const int b = p0.yoff + m2;
                        if (hdef.count({a, b})) S(fmt("dxp_%d = fma(%s_%d, h_%d_%d, dxp_%d);", a, yname, b, a, b, a));
                    }
                }
            }
            S.ind--;
            S("}");
        }
    }

    // ------------------------------------------------------------------ backward edge kernel
    void emit_edge_group(Src& S, int g) const {
        const std::vector<int>& paths = P->groups[g];
        const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
        std::vector<int> outs;
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            for (int m = 0; m < 2 * p.l3 + 1; ++m) outs.push_back(p.ooff + m);
        }
        S(fmt("__device__ __forceinline__ void edge_group%d(int rl, int seg, int lane_in_seg, bool valid, int r_e0, int r_e1,", g));
        S(fmt("    int nchunks, long long r, int u, const int* __restrict__ src, const %s* __restrict__ x,", T.c_str()));
        S(fmt("    const %s* __restrict__ Y, const %s* __restrict__ w, const %s* __restrict__ gout,", T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    %s* __restrict__ dY, %s* __restrict__ dw, %s* __restrict__ dx, %s* sred, const int* s_e0, const int* s_e1,",
              T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    %s* __restrict__ dxe) {", T.c_str()));
        S.ind++;
        S(fmt("const %s* __restrict__ grow = gout + ((size_t)(valid ? r : 0) * UVU_U + u) * UVU_DO;", T.c_str()));
        for (int k : outs) S(fmt("const %s gv_%d = valid ? __ldg(grow + %d) : (%s)0;", T.c_str(), k, k, T.c_str()));
        S("#pragma unroll 1");
        S("for (int c = 0; c < nchunks; ++c) {");
        S.ind++;
        S("#pragma unroll 1");
        S("for (int j = 0; j < UVU_CH; ++j) {");
        S.ind++;
        S("const int e = r_e0 + c * UVU_CH + j;");
        S("const bool active = valid && e < r_e1;");
        for (int k : yn) S(fmt("%s dyp_%d = 0;", T.c_str(), k));
        S("if (active) {");
        S.ind++;
        S("const int s = __ldg(src + e);");
        emit_row_loads(S, "xv", "x + ((size_t)s * UVU_U + u) * UVU_DX", P->Dx, xn);
        emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        S("const " + T + "* __restrict__ we = w + (size_t)e * (UVU_P * UVU_U) + u;");
        S(T + "* __restrict__ dwe = dw + (size_t)e * (UVU_P * UVU_U) + u;");
        for (int pi : paths) S(fmt("const %s wv_%d = __ldg(we + %d * UVU_U);", T.c_str(), pi, pi));
        for (int k : xn) S(fmt("%s dxp_%d = 0;", T.c_str(), k));
        emit_products(S, paths);
        auto gval = [](int k) { return fmt("gv_%d", k); };
        S("if (dw) {");
        S.ind++;
        emit_bwd_pairs(S, paths, true, false, false, gval);
        S.ind--;
        S("}");
        emit_bwd_pairs(S, paths, false, true, true, gval);
        // atomic dx scatter
        S("if (dx) {");
        S.ind++;
        S(T + "* __restrict__ dxr = dx + ((size_t)s * UVU_U + u) * UVU_DX;");
        if (!f64 && P->Dx % 4 == 0) {
            std::set<int> chunks;
            for (int k : xn) chunks.insert(k / 4);
            for (int c : chunks) {
                std::string v[4];
                for (int i = 0; i < 4; ++i) v[i] = xn.count(4 * c + i) ? fmt("dxp_%d", 4 * c + i) : "0.0f";
                S(fmt("red_add_v4(dxr + %d, %s, %s, %s, %s);", 4 * c, v[0].c_str(), v[1].c_str(), v[2].c_str(), v[3].c_str()));
            }
        } else {
            for (int k : xn) S(fmt("atomicAdd(dxr + %d, dxp_%d);", k, k));
        }
        S.ind--;
        S("}");
        if (P->groups.size() == 1) emit_dx_edge_store(S, xn, 1);
        S.ind--;
        S("}");  // active
        // reduce the dY partials over the channels of this segment
        S("if (dY) {");
        S.ind++;
        for (int k : yn) {
            S(fmt("#pragma unroll"));
            S(fmt("for (int o = UVU_SEGW / 2; o > 0; o >>= 1) dyp_%d += __shfl_xor_sync(0xffffffffu, dyp_%d, o);", k, k));
        }
        S("if (lane_in_seg == 0) {");
        S.ind++;
        S(T + "* sr = sred + ((size_t)(rl * UVU_SEGS + seg) * UVU_CH + j) * UVU_DY;");
        for (int k = 0; k < P->Dy; ++k) {
            if (yn.count(k)) S(fmt("sr[%d] = dyp_%d;", k, k));
            else S(fmt("sr[%d] = 0;", k));
        }
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S.ind--;
        S("}");  // j
        S("block_sync();");
        S("if (dY) {");
        S.ind++;
        S("for (int it = threadIdx.x; it < UVU_RPB * UVU_CH * UVU_DY; it += UVU_TPB) {");
        S.ind++;
        S("const int k = it % UVU_DY, jj = (it / UVU_DY) % UVU_CH, r2 = it / (UVU_DY * UVU_CH);");
        S("const int e = s_e0[r2] + c * UVU_CH + jj;");
        S("if (e < s_e1[r2]) {");
        S.ind++;
        S(T + " acc = 0;");
        S("#pragma unroll");
        S("for (int sg = 0; sg < UVU_SEGS; ++sg) acc += sred[((size_t)(r2 * UVU_SEGS + sg) * UVU_CH + jj) * UVU_DY + k];");
        S("dY[(size_t)e * UVU_DY + k] = acc;");
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S("block_sync();");
        S.ind--;
        S("}");  // c
        S.ind--;
        S("}");
    }

    // ================================================================== double backward (HVP)
    // With T = <g, F(x, Y, w)> multilinear, the gradients of L2 = <ax,dx> + <aY,dY> + <aw,dw>
    // are forward / VJP contractions with one argument substituted ("Receiver-streaming
    // convolutions ...", results table, HVP column; "An Efficient Sparse Kernel Generator ...",
    // abstract, higher partial derivatives):
    //   dL2/dg = F(ax,Y,w) + F(x,aY,w) + F(x,Y,aw)          -> uvu_hvp_fwd (receiver-stationary)
    //   dL2/dw = dw(x<-ax) + dw(Y<-aY)                       -> uvu_hvp_edge
    //   dL2/dY = dY(x<-ax) + dY(w<-aw)                       -> uvu_hvp_edge
    //   dL2/dx = dx(Y<-aY) + dx(w<-aw)  per edge, then the sender-stationary reduction
    // Absent cotangents are marked in the bit mask hm (1 = ax, 2 = aY, 4 = aw) and read as zero.

    // Declares pre_k = 0 for k in `need`, then loads them from `base` when `cond` holds.
    void emit_row_loads_masked(Src& S, const std::string& pre, const std::string& base, int width,
                               const std::set<int>& need, const std::string& cond, bool global = true) const {
        for (int k : need) S(fmt("%s %s_%d = 0;", T.c_str(), pre.c_str(), k));
        S("if (" + cond + ") {");
        S.ind++;
        emit_row_loads(S, pre + "l", base, width, need, global);
        for (int k : need) S(fmt("%s_%d = %sl_%d;", pre.c_str(), k, pre.c_str(), k));
        S.ind--;
        S("}");
    }

    // q_a_b = ax_a y_b + x_a ay_b  (the mixed products of the substituted forward terms)
    void emit_mixed_products(Src& S, const std::vector<int>& paths, const char* name) const {
        std::set<std::pair<int, int>> q;
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            for (const Nz& z : p.nz) q.insert({p.xoff + z.m1, p.yoff + z.m2});
        }
        for (auto& ab : q)
            S(fmt("const %s %s_%d_%d = fma(axv_%d, yv_%d, xv_%d * ayv_%d);", T.c_str(), name, ab.first, ab.second,
                  ab.first, ab.second, ab.first, ab.second));
    }

    void emit_hvp_edge_loads(Src& S, const std::vector<int>& paths) const {
        const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
        S("const int s = __ldg(src + e);");
        emit_row_loads(S, "xv", "x + ((size_t)s * UVU_U + u) * UVU_DX", P->Dx, xn);
        emit_row_loads_masked(S, "axv", "ax + ((size_t)s * UVU_U + u) * UVU_DX", P->Dx, xn, "hm & 1");
        emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        emit_row_loads_masked(S, "ayv", "aY + (size_t)e * UVU_DY", P->Dy, yn, "hm & 2");
        S("const " + T + "* __restrict__ we = w + (size_t)e * (UVU_P * UVU_U) + u;");
        for (int pi : paths) S(fmt("const %s wv_%d = __ldg(we + %d * UVU_U);", T.c_str(), pi, pi));
        for (int pi : paths) S(fmt("%s awv_%d = 0;", T.c_str(), pi));
        S("if (hm & 4) {");
        S("  const " + T + "* __restrict__ awe = aw + (size_t)e * (UVU_P * UVU_U) + u;");
        for (int pi : paths) S(fmt("  awv_%d = __ldg(awe + %d * UVU_U);", pi, pi));
        S("}");
    }

    // Per-edge part of dL2/dg: F(ax,Y,w) + F(x,aY,w) through the mixed products, plus F(x,Y,aw).
    void emit_hvp_fwd_edge(Src& S, const std::vector<int>& paths) const {
        emit_mixed_products(S, paths, "qm");
        emit_products(S, paths);
        for (int pi : paths) {
            const PathInfo& p = P->paths[pi];
            S("{");
            S.ind++;
            emit_t(S, pi, "qm", "tm");
            emit_t(S, pi, "q", "t");
            for (int m3 = 0; m3 < 2 * p.l3 + 1; ++m3)
                S(fmt("acc_%d = fma(wv_%d, tm_%d_%d, fma(awv_%d, t_%d_%d, acc_%d));", p.ooff + m3, pi, pi, m3, pi, pi, m3,
                      p.ooff + m3));
            S.ind--;
            S("}");
        }
    }

    void emit_hvp_fwd_group(Src& S, int g) const {
        const std::vector<int>& paths = P->groups[g];
        std::vector<int> outs;
        for (int pi : paths)
            for (int m = 0; m < 2 * P->paths[pi].l3 + 1; ++m) outs.push_back(P->paths[pi].ooff + m);
        S(fmt("__device__ __forceinline__ void hvp_fwd_group%d(int e0, int e1, int u, int hm, const int* __restrict__ src,", g));
        S(fmt("    const %s* __restrict__ x, const %s* __restrict__ Y, const %s* __restrict__ w, const %s* __restrict__ ax,",
              T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    const %s* __restrict__ aY, const %s* __restrict__ aw, %s* __restrict__ orow) {", T.c_str(), T.c_str(), T.c_str()));
        S.ind++;
        for (int k : outs) S(fmt("%s acc_%d = 0;", T.c_str(), k));
        S("#pragma unroll 1");
        S("for (int e = e0; e < e1; ++e) {");
        S.ind++;
        emit_hvp_edge_loads(S, paths);
        emit_hvp_fwd_edge(S, paths);
        S.ind--;
        S("}");
        for (int k : outs) S(fmt("orow[%d] = acc_%d;", k, k));
        S.ind--;
        S("}");
    }

    void emit_hvp_edge_group(Src& S, int g) const {
        const std::vector<int>& paths = P->groups[g];
        const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
        std::vector<int> outs;
        for (int pi : paths)
            for (int m = 0; m < 2 * P->paths[pi].l3 + 1; ++m) outs.push_back(P->paths[pi].ooff + m);
        S(fmt("__device__ __forceinline__ void hvp_edge_group%d(int rl, int seg, int lane_in_seg, bool valid, int r_e0, int r_e1,", g));
        S(fmt("    int nchunks, long long r, int u, int hm, const int* __restrict__ src, const %s* __restrict__ x,", T.c_str()));
        S(fmt("    const %s* __restrict__ Y, const %s* __restrict__ w, const %s* __restrict__ gout,", T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    const %s* __restrict__ ax, const %s* __restrict__ aY, const %s* __restrict__ aw,", T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    %s* __restrict__ dY, %s* __restrict__ dw, %s* __restrict__ dx, %s* __restrict__ dxe, %s* sred,",
              T.c_str(), T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        S("    const int* s_e0, const int* s_e1) {");
        S.ind++;
        S(fmt("const %s* __restrict__ grow = gout + ((size_t)(valid ? r : 0) * UVU_U + u) * UVU_DO;", T.c_str()));
        for (int k : outs) S(fmt("const %s gv_%d = valid ? __ldg(grow + %d) : (%s)0;", T.c_str(), k, k, T.c_str()));
        S("#pragma unroll 1");
        S("for (int c = 0; c < nchunks; ++c) {");
        S.ind++;
        S("#pragma unroll 1");
        S("for (int j = 0; j < UVU_CH; ++j) {");
        S.ind++;
        S("const int e = r_e0 + c * UVU_CH + j;");
        S("const bool active = valid && e < r_e1;");
        for (int k : yn) S(fmt("%s dyp_%d = 0;", T.c_str(), k));
        S("if (active) {");
        S.ind++;
        emit_hvp_edge_loads(S, paths);
        S(T + "* __restrict__ dwe = dw + (size_t)e * (UVU_P * UVU_U) + u;");
        for (int k : xn) S(fmt("%s dxp_%d = 0;", T.c_str(), k));
        auto gval = [](int k) { return fmt("gv_%d", k); };
        S("if (dw) {");
        S.ind++;
        emit_mixed_products(S, paths, "q");
        emit_bwd_pairs(S, paths, true, false, false, gval);
        S.ind--;
        S("}");
        emit_bwd_pairs(S, paths, false, true, true, gval, "axv", "ayv", "wv");
        emit_bwd_pairs(S, paths, false, true, true, gval, "xv", "yv", "awv");
        S("if (dx) {");
        S.ind++;
        S(T + "* __restrict__ dxr = dx + ((size_t)s * UVU_U + u) * UVU_DX;");
        emit_dx_atomics(S, xn);
        S.ind--;
        S("}");
        if (P->groups.size() == 1) emit_dx_edge_store(S, xn, 1);
        S.ind--;
        S("}");  // active
        S("if (dY) {");
        S.ind++;
        for (int k : yn) {
            S("#pragma unroll");
            S(fmt("for (int o = UVU_SEGW / 2; o > 0; o >>= 1) dyp_%d += __shfl_xor_sync(0xffffffffu, dyp_%d, o);", k, k));
        }
        S("if (lane_in_seg == 0) {");
        S.ind++;
        S(T + "* sr = sred + ((size_t)(rl * UVU_SEGS + seg) * UVU_CH + j) * UVU_DY;");
        for (int k = 0; k < P->Dy; ++k) {
            if (yn.count(k)) S(fmt("sr[%d] = dyp_%d;", k, k));
            else S(fmt("sr[%d] = 0;", k));
        }
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S.ind--;
        S("}");  // j
        S("block_sync();");
        S("if (dY) {");
        S.ind++;
        S("for (int it = threadIdx.x; it < UVU_RPB * UVU_CH * UVU_DY; it += UVU_TPB) {");
        S.ind++;
        S("const int k = it % UVU_DY, jj = (it / UVU_DY) % UVU_CH, r2 = it / (UVU_DY * UVU_CH);");
        S("const int e = s_e0[r2] + c * UVU_CH + jj;");
        S("if (e < s_e1[r2]) {");
        S.ind++;
        S(T + " acc = 0;");
        S("#pragma unroll");
        S("for (int sg = 0; sg < UVU_SEGS; ++sg) acc += sred[((size_t)(r2 * UVU_SEGS + sg) * UVU_CH + jj) * UVU_DY + k];");
        S("dY[(size_t)e * UVU_DY + k] = acc;");
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S("block_sync();");
        S.ind--;
        S("}");  // c
        S.ind--;
        S("}");
    }

    void emit_hvp_kernels(Src& S) const {
        const int NG = int(P->groups.size());
        no_identity = true;
        for (int g = 0; g < NG; ++g) emit_hvp_fwd_group(S, g);
        for (int g = 0; g < NG; ++g) emit_hvp_edge_group(S, g);
        no_identity = false;
        const char* t = T.c_str();
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_TPB) uvu_hvp_fwd(long long N, const int* __restrict__ off,"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y, const %s* __restrict__ w,", t, t, t));
        S(fmt("    const %s* __restrict__ ax, const %s* __restrict__ aY, const %s* __restrict__ aw, int hm, %s* __restrict__ out) {", t, t, t, t));
        S("  const int u = threadIdx.x % UVU_UP;");
        S("  const int g = (threadIdx.x / UVU_UP) % UVU_G;");
        S("  const long long r = (long long)blockIdx.x * UVU_RPB + threadIdx.x / (UVU_UP * UVU_G);");
        S("  if (r >= N || u >= UVU_U) return;");
        S("  const int e0 = __ldg(off + r), e1 = __ldg(off + r + 1);");
        S(fmt("  %s* orow = out + ((size_t)r * UVU_U + u) * UVU_DO;", t));
        for (int g = 0; g < NG; ++g)
            S(fmt("  %sif (g == %d) hvp_fwd_group%d(e0, e1, u, hm, src, x, Y, w, ax, aY, aw, orow);", g ? "else " : "", g, g));
        S("}");
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_TPB) uvu_hvp_edge(long long N, const int* __restrict__ off,"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y, const %s* __restrict__ w,", t, t, t));
        S(fmt("    const %s* __restrict__ gout, const %s* __restrict__ ax, const %s* __restrict__ aY, const %s* __restrict__ aw,", t, t, t, t));
        S(fmt("    int hm, %s* __restrict__ dY, %s* __restrict__ dw, %s* __restrict__ dx, %s* __restrict__ dxe) {", t, t, t, t));
        S("  extern __shared__ __align__(16) unsigned char smem_raw[];");
        S(fmt("  %s* sred = reinterpret_cast<%s*>(smem_raw);", t, t));
        S("  __shared__ int s_e0[UVU_RPB], s_e1[UVU_RPB], s_nch;");
        S("  const int u = threadIdx.x % UVU_UP;");
        S("  const int g = (threadIdx.x / UVU_UP) % UVU_G;");
        S("  const int rl = threadIdx.x / (UVU_UP * UVU_G);");
        S("  const long long r = (long long)blockIdx.x * UVU_RPB + rl;");
        S("  const bool rvalid = r < N;");
        S("  const bool valid = rvalid && u < UVU_U;");
        S("  if (threadIdx.x == 0) s_nch = 0;");
        S("  __syncthreads();");
        S("  if (threadIdx.x % (UVU_UP * UVU_G) == 0) {");
        S("    const int a = rvalid ? __ldg(off + r) : 0, b = rvalid ? __ldg(off + r + 1) : 0;");
        S("    s_e0[rl] = a; s_e1[rl] = b;");
        S("    atomicMax(&s_nch, (b - a + UVU_CH - 1) / UVU_CH);");
        S("  }");
        S("  __syncthreads();");
        S("  const int nchunks = s_nch;");
        S("  const int seg = g * ((UVU_UP + 31) / 32) + u / 32;");
        S("  const int lane_in_seg = u % UVU_SEGW;");
        for (int g = 0; g < NG; ++g)
            S(fmt("  %sif (g == %d) hvp_edge_group%d(rl, seg, lane_in_seg, valid, s_e0[rl], s_e1[rl], nchunks, r, u, hm, src, x, Y, w, gout, ax, aY, aw, dY, dw, dx, dxe, sred, s_e0, s_e1);",
                  g ? "else " : "", g, g));
        S("}");
    }

    // ------------------------------------------------------------------ sender-stationary dx
    void emit_dx_kernel(Src& S) const {
        std::vector<int> all;
        for (int p = 0; p < P->P; ++p) all.push_back(p);
        const std::set<int> xn = x_needed(all), yn = y_needed(all);
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_DX_TPB) uvu_bwd_dx(long long N, const int* __restrict__ soff,"));
        S(fmt("    const int* __restrict__ seid, const int* __restrict__ srecv, const %s* __restrict__ Y,", T.c_str()));
        S(fmt("    const %s* __restrict__ w, const %s* __restrict__ gout, %s* __restrict__ dx) {", T.c_str(), T.c_str(), T.c_str()));
        S.ind++;
        S("const int u = threadIdx.x % UVU_UP;");
        S("const long long sn = (long long)blockIdx.x * UVU_SPB + threadIdx.x / UVU_UP;");
        S("if (sn >= N || u >= UVU_U) return;");
        S("const int k0 = __ldg(soff + sn), k1 = __ldg(soff + sn + 1);");
        for (int k : xn) S(fmt("%s dxp_%d = 0;", T.c_str(), k));
        S("#pragma unroll 1");
        S("for (int kk = k0; kk < k1; ++kk) {");
        S.ind++;
        S("const int e = __ldg(seid + kk);");
        S("const int r = __ldg(srecv + kk);");
        emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        S("const " + T + "* __restrict__ we = w + (size_t)e * (UVU_P * UVU_U) + u;");
        S("const " + T + "* __restrict__ grow = gout + ((size_t)r * UVU_U + u) * UVU_DO;");
        for (int pi : all) S(fmt("const %s wv_%d = __ldg(we + %d * UVU_U);", T.c_str(), pi, pi));
        auto gval = [](int k) { return fmt("__ldg(grow + %d)", k); };
        emit_bwd_pairs(S, all, false, false, true, gval);
        S.ind--;
        S("}");
        S(T + "* __restrict__ dxr = dx + ((size_t)sn * UVU_U + u) * UVU_DX;");
        for (int k = 0; k < P->Dx; ++k) S(fmt("dxr[%d] = %s;", k, xn.count(k) ? fmt("dxp_%d", k).c_str() : "0"));
        S.ind--;
        S("}");
    }

    // ================================================================== pipelined kernels
    // One producer warp streams the per-edge operands of each owner into a ring of NST shared
    // memory stages with cp.async.bulk (completion counted on an mbarrier per stage); the
    // consumer warps compute from shared memory and release the stage on a second mbarrier.
    // Owners (receivers or senders) are assigned round-robin to persistent CTAs.
    // Every wait is bounded (about two seconds on the global timer): on expiry the kernel sets
    // a bit in uvu_status_word, skips the remaining work and returns.

    // Per-edge operand sizes in bytes.
    size_t wbytes() const { return size_t(P->P) * P->U * P->elem(); }
    size_t xbytes() const { return size_t(P->U) * P->Dx * P->elem(); }
    size_t ybytes() const { return size_t(P->Dy) * P->elem(); }

    // Release of a stage by the consumer warps.  The stage's shared memory was read through the
    // generic proxy and the producer's next cp.async.bulk writes it through the async proxy, so
    // every lane fences its reads (a CTA fence plus the generic->async proxy fence) before its
    // warp's single arrival on the stage's "empty" barrier.  Without the fences the next copy
    // was observed to overwrite data a warp had not finished reading.
    // UVU_DBG_RELEASE (a debugging switch): 1 = per-thread arrival without fences,
    // 3 = proxy fence only.
    int release_mode() const {
        const char* e = std::getenv("UVU_DBG_RELEASE");
        return e ? std::atoi(e) : 0;
    }
    void emit_release(Src& S, const char* pre) const {
        const int m = release_mode();
        if (m == 1) {
            S(fmt("mbar_arrive(sbase + %s_BAR + 8u * (%s_NST + st));", pre, pre));
            return;
        }
        if (m != 3) S("__threadfence_block();");
        S("asm volatile(\"fence.proxy.async.shared::cta;\" ::: \"memory\");");
        S("__syncwarp();");
        S(fmt("if (lane == 0) mbar_arrive(sbase + %s_BAR + 8u * (%s_NST + st));", pre, pre));
    }
    // Arrival count of a stage's "empty" barrier: one per consumer warp (or per consumer thread
    // under the per-thread debugging release).
    const char* empty_count(const char* ncw, const char* nct) const { return release_mode() == 1 ? nct : ncw; }
    void emit_pipe_helpers(Src& S) const {
        S(R"(__device__ unsigned int uvu_status_word;
#define UVU_DEV_TIMEOUT 1u
__device__ __forceinline__ unsigned smem_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(unsigned b, unsigned n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned b, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(b) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned b, unsigned parity) {
  unsigned ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
               : "=r"(ok) : "r"(b), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Slow path of a bounded wait: gives up after about two seconds and records the timeout.
__device__ __noinline__ bool mbar_wait_slow(unsigned b, unsigned parity) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_test(b, parity)) return true;
    if (global_ns() - t0 > 2000000000ull) {
      atomicOr(&uvu_status_word, UVU_DEV_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait(unsigned b, unsigned parity) {
  return mbar_test(b, parity) || mbar_wait_slow(b, parity);
}
__device__ __forceinline__ void bulk_g2s(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// Bulk copy shared -> global (the async proxy reads [src, src + bytes) of this CTA's shared
// memory); completion tracked per thread by bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* dst, unsigned src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" :: "l"(dst), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the source reads of every committed group are done (the shared memory may be reused)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed group is complete (its global writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Asks the memory system to bring [src, src + bytes) into L2 ahead of its use (no completion
// to wait for; the later bulk copy to shared memory then hits in L2).
__device__ __forceinline__ void prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}
// Barrier among the consumer warps only (the producer warp never takes part).
__device__ __forceinline__ void consumer_sync() { asm volatile("barrier.sync 1, %0;" :: "r"(UVU_NCT) : "memory"); })");
    }

    // Stage layout of the receiver-ordered kernels (forward and edge backward).
    struct RecvPipe {
        int ch = 1, nst = 2;
        int pf = 0;  // L2 prefetch distance in chunks (0 = none; prefetching measured slower)
        bool xbulk = false, ybulk = false;
        int odp = 0;  // row stride (elements) of the staged output block, 0 = not staged
        bool ovec = false;  // staged block copied out with 16-byte vectors
        bool gst = false;  // the receiver's d_out block is bulk-copied into shared memory
        // gsm (with gst, plain edge kernel): each d_out value is read from the staged block where
        // it is used, and the block is released when the receiver is done, instead of the row
        // being copied into registers at the receiver start (frees D_out registers per thread)
        bool gsm = false;
        bool dual = false;  // double backward: the stage also holds the cotangent rows aw, ax, aY
        bool tp = false;    // batched tensor product: sample b is receiver b with the one edge b, sender b
        bool wsh = false;   // weights [P][U] shared by the batch: not staged, read once per sample
        size_t aw_off = 0, ax_off = 0, ay_off = 0;
        size_t w_off = 0, x_off = 0, y_off = 0, stage = 0, bar_off = 0, part_off = 0, xpart_off = 0, out_off = 0, total = 0;
        size_t g_off = 0, gbytes = 0;
        size_t dacc_off = 0;  // fp64 dw accumulators [P][U_pad] of the batch-shared-weight edge kernel
        // edge kernel, one register group, UVU_PIPE_LASTWARP=1 (a tuning switch): the per-stage dY
        // partials are summed by the last warp to finish the stage (an arrival counter per buffer,
        // three buffers) instead of after a barrier of all consumer warps.  Off by default: it
        // measured slower (MACE-medium edge kernel 0.897 vs 0.862 ms); the barrier keeps the warps
        // in step over the shared stages.
        bool lastwarp = false;
        // dY's cross-lane sum through a per-warp shared-memory tile (fp32, 9..16 SH components)
        // instead of the shuffle transpose-reduce
        bool dyt = false;
        size_t dyt_off = 0;
        int nbuf = 2;
        size_t cnt_off = 0;
        size_t tx_per_edge = 0;
    };
    static size_t a16(size_t v) { return (v + 15) / 16 * 16; }

    // A forward-type pipe (no per-stage partials) whose stages hold one edge each gets a third
    // stage when that keeps as many blocks resident as two stages (capped at `cap`): with
    // one-edge stages and one or two blocks per SM, two stages keep too few bytes in flight
    // (measured: wide forward 1.95 -> 1.61 ms, MACE-large 0.86 -> 0.83 ms).  UVU_PIPE_NST
    // overrides it.
    RecvPipe fwd_pipe(int ncw, int cap, bool stage_out, bool dual = false, bool tp = false, bool wsh = false) const {
        RecvPipe R = recv_pipe(false, ncw, stage_out, 0, false, dual, tp, wsh);
        if (R.ch != 1 || std::getenv("UVU_PIPE_NST")) return R;
        RecvPipe R3 = recv_pipe(false, ncw, R.odp != 0, 1, false, dual, tp, wsh, 3);
        return minb(R3.total) >= std::min(minb(R.total), cap) ? R3 : R;
    }

    RecvPipe recv_pipe(bool with_partials, int ncw, bool stage_out = false, int ch = 0, bool stage_g = false,
                       bool dual = false, bool tp = false, bool wsh = false, int nst_req = 0) const {
        RecvPipe R;
        R.dual = dual;
        R.tp = tp;
        R.wsh = wsh;
        R.xbulk = xbytes() % 16 == 0;
        R.ybulk = ybytes() % 16 == 0;
        const int NG = int(P->groups.size());
        const size_t wb = wsh ? 0 : wbytes();  // staged weight bytes per edge
        const size_t pe = std::max<size_t>(16, (wb + (R.xbulk ? xbytes() : 0) + (R.ybulk ? ybytes() : 0)) * (dual ? 2 : 1));
        const bool chosen = ch > 0 || std::getenv("UVU_PIPE_CH") || tp;
        R.ch = ch > 0 ? ch : int(std::max<size_t>(1, std::min<size_t>(8, 32768 / pe)));
        if (const char* e = std::getenv("UVU_PIPE_CH")) R.ch = std::max(1, std::atoi(e));
        if (tp) R.ch = 1;  // one edge per receiver
        const size_t stage = std::max<size_t>(16, (a16(R.ch * wb) + (R.xbulk ? a16(R.ch * xbytes()) : 0) +
                                                   (R.ybulk ? a16(R.ch * ybytes()) : 0)) * (dual ? 2 : 1));
        // per-stage partial sums of the edge kernel: dY over warps, dx over register groups
        R.lastwarp = with_partials && NG == 1 && std::getenv("UVU_PIPE_LASTWARP") &&
                     std::atoi(std::getenv("UVU_PIPE_LASTWARP")) != 0;
        R.nbuf = R.lastwarp ? 3 : 2;
        const size_t dyp = with_partials ? a16(size_t(R.nbuf) * ncw * R.ch * P->Dy * P->elem()) + (R.lastwarp ? 16 : 0) : 0;
        const size_t dxp = (with_partials && NG > 1) ? a16(2 * size_t(NG) * R.ch * P->U_pad * P->Dx * P->elem()) : 0;
        // Two stages: with several blocks resident per SM, one stage of look-ahead per block keeps
        // enough bytes in flight, and the smaller footprint lets more blocks (warps) reside.
        R.nst = nst_req > 0 ? nst_req : 2;
        if (const char* e = std::getenv("UVU_PIPE_NST")) R.nst = std::max(2, std::atoi(e));
        if (const char* e = std::getenv("UVU_PIPE_PF")) R.pf = std::max(0, std::atoi(e));
        R.w_off = 0;
        R.aw_off = dual ? a16(R.ch * wbytes()) : 0;
        R.x_off = (dual ? 2 : 1) * a16(R.ch * wb);
        R.ax_off = R.x_off + ((dual && R.xbulk) ? a16(R.ch * xbytes()) : 0);
        R.y_off = R.x_off + (R.xbulk ? (dual ? 2 : 1) * a16(R.ch * xbytes()) : 0);
        R.ay_off = R.y_off + ((dual && R.ybulk) ? a16(R.ch * ybytes()) : 0);
        R.stage = stage;
        R.bar_off = R.nst * stage;
        // The edge kernel's d_out block (U x D_out, contiguous) arrives by one bulk copy per
        // receiver into a buffer of its own, with a full/empty barrier pair after the stages'.
        R.gbytes = size_t(P->U) * P->Do * P->elem();
        R.gst = stage_g && R.gbytes % 16 == 0;
        R.part_off = R.bar_off + 16 * R.nst + (R.gst ? 16 : 0);
        R.xpart_off = R.part_off + dyp;
        R.cnt_off = R.part_off + dyp - (R.lastwarp ? 16 : 0);
        R.out_off = R.xpart_off + dxp;
        // The receiver's output block out[r] (U x D_out, contiguous in global memory) is staged in
        // shared memory so that it leaves the block as coalesced row writes instead of one
        // D_out-strided store per thread and output component.  Rows are padded to an odd stride
        // so that the per-thread row writes fall in distinct banks.
        if (stage_out) {
            R.odp = P->Do % 2 ? P->Do : P->Do + 1;
            R.ovec = R.odp == P->Do && (size_t(P->U) * P->Do * P->elem()) % 16 == 0;
        }
        R.total = R.out_off + (stage_out ? a16(size_t(P->U) * R.odp * P->elem()) : 0);
        R.g_off = R.total;
        if (R.gst) R.total += a16(R.gbytes);
        R.dacc_off = R.total;
        if (wsh && with_partials && !f64) R.total += a16(size_t(P->P) * P->U_pad * 8);
        // measured: MACE-large VJP 2.514 -> 2.442 ms, wide 5.183 -> 5.061 ms; slower on MACE-medium
        // (edge kernel 0.776 -> 0.790 ms) and in the double backward (1.455 -> 1.527 ms), so only the
        // plain edge kernels with wide output rows (fp32, D_out > 64) take it
        R.dyt = with_partials && !f64 && !dual && !tp && P->Do > 64 && P->Dy > 8 && P->Dy <= 16 && dy_smem_enabled();
        if (R.dyt) {
            R.dyt_off = R.total;
            R.total += a16(size_t(ncw) * kDytWords * 4);
        }
        R.tx_per_edge = wb + (R.xbulk ? xbytes() : 0) + (R.ybulk ? ybytes() : 0);
        // With a receiver block staged, shorter stages keep three blocks resident per SM where
        // the default chunk would leave fewer (more warps beat a longer look-ahead per block).
        if ((stage_out || R.gst) && !chosen && R.ch > 1 && minb(R.total) < 3)
            return recv_pipe(with_partials, ncw, stage_out, R.ch - 1, stage_g, dual, tp, wsh, nst_req);
        // a staged block that does not fit next to the stages is not staged
        if (R.total > 227 * 1024 && R.gst) return recv_pipe(with_partials, ncw, stage_out, ch, false, dual, tp, wsh, nst_req);
        if (R.total > 227 * 1024 && stage_out) return recv_pipe(with_partials, ncw, false, ch, stage_g, dual, tp, wsh, nst_req);
        return R;
    }

    // cap / eff: the kernel's entries in its register-budget tables (blocks per SM allowed, used)
    void emit_recv_pipe_defines(Src& S, const RecvPipe& R, const char* pre, int& cap, int& eff) const {
        S(fmt("#define %s_CH %d", pre, R.ch));
        S(fmt("#define %s_NST %d", pre, R.nst));
        S(fmt("#define %s_STAGE %zu", pre, R.stage));
        S(fmt("#define %s_XOFF %zu", pre, R.x_off));
        S(fmt("#define %s_YOFF %zu", pre, R.y_off));
        S(fmt("#define %s_BAR %zu", pre, R.bar_off));
        S(fmt("#define %s_PART %zu", pre, R.part_off));
        S(fmt("#define %s_XPART %zu", pre, R.xpart_off));
        S(fmt("#define %s_TX %zu", pre, R.tx_per_edge));
        S(fmt("#define %s_OBUF %zu", pre, R.out_off));
        S(fmt("#define %s_GBUF %zu", pre, R.g_off));
        S(fmt("#define %s_GBAR %zu", pre, R.bar_off + 16 * R.nst));
        S(fmt("#define %s_GBYTES %zu", pre, R.gbytes));
        S(fmt("#define %s_DACC %zu", pre, R.dacc_off));
        if (R.dyt) S(fmt("#define %s_DYT %zu", pre, R.dyt_off));
        if (R.lastwarp) {
            S(fmt("#define %s_CNT %zu", pre, R.cnt_off));
            S(fmt("#define %s_NBUF %d", pre, R.nbuf));
        }
        S(fmt("#define %s_AWOFF %zu", pre, R.aw_off));
        S(fmt("#define %s_AXOFF %zu", pre, R.ax_off));
        S(fmt("#define %s_AYOFF %zu", pre, R.ay_off));
        S(fmt("#define %s_ODP %d", pre, R.odp));
        const int mb = std::min(minb(R.total), cap);
        eff = mb;
        S(fmt("#define %s_MINB %d", pre, mb));
    }
    // Blocks per SM the shared-memory footprint allows (capped at 4); UVU_PIPE_MINB (a tuning
    // switch) lowers the cap.
    static int minb(size_t smem) {
        size_t cap = 4;
        if (const char* e = std::getenv("UVU_PIPE_MINB")) cap = size_t(std::max(1, std::atoi(e)));
        return int(std::max<size_t>(1, std::min<size_t>(cap, (227 * 1024) / (smem + 1024))));
    }

    // Producer for the receiver-ordered kernels: w block of the chunk (one copy, the receiver's
    // edges are contiguous), Y block (one copy), x row of each edge's sender (one copy each).
    // The sender ids of the next chunk and the offsets of the next receiver are loaded one step
    // ahead, before the current chunk's copies are issued: the copies are asm statements with a
    // memory clobber, so a load placed after one of them would wait its full latency in line.
    // Receiver offsets and sender ids: from the CSR, or the identity for the batched tensor
    // product (sample b = receiver b with the single edge b from sender b).
    static std::string off_at(const RecvPipe& R, const std::string& r) {
        return R.tp ? "(int)(" + r + ")" : "__ldg(off + " + r + ")";
    }
    static std::string src_at(const RecvPipe& R, const std::string& e) {
        return R.tp ? "(" + e + ")" : "__ldg(src + " + e + ")";
    }

    void emit_recv_producer(Src& S, const RecvPipe& R, const char* pre, const char* name) const {
        const int CH = R.ch;
        S(fmt("__device__ __noinline__ void %s(long long N, const int* __restrict__ off, const int* __restrict__ src,", name));
        S(fmt("    const %s* __restrict__ x, const %s* __restrict__ Y, const %s* __restrict__ w, const %s* __restrict__ gout,",
              T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        if (R.dual)
            S(fmt("    const %s* __restrict__ ax, const %s* __restrict__ aY, const %s* __restrict__ aw, int hm,", T.c_str(), T.c_str(),
                  T.c_str()));
        S("    unsigned sbase) {");
        S.ind++;
        if (R.dual)  // bytes per edge with the cotangent rows that are present (mask hm: 1 = ax, 2 = aY, 4 = aw)
            S(fmt("const unsigned txe = %s_TX + ((hm & 4) ? %zuu : 0u) + ((hm & 2) ? %zuu : 0u) + ((hm & 1) ? %zuu : 0u);", pre,
                  wbytes(), R.ybulk ? ybytes() : size_t(0), R.xbulk ? xbytes() : size_t(0)));
        S("unsigned c = 0;");
        if (R.gst) S("unsigned kg = 0;  // d_out blocks issued");
        if (R.gst) S("bool fresh = true;  // no chunk of receiver r issued yet");
        S("bool dead = false;");
        S("const long long G = gridDim.x;");
        S("long long r = blockIdx.x;");
        S("int eb = 0, e1 = 0, nb = 0, n1 = 0;");
        S("if (r < N) { eb = " + off_at(R, "r") + "; e1 = " + off_at(R, "r + 1") + "; }");
        S("if (r + G < N) { nb = " + off_at(R, "r + G") + "; n1 = " + off_at(R, "r + G + 1") + "; }");
        for (int j = 0; j < CH; ++j) S(fmt("int sv%d = (%d < e1 - eb) ? %s : 0;", j, j, src_at(R, fmt("eb + %d", j)).c_str()));
        S("while (r < N && !dead) {");
        S.ind++;
        S("if (eb >= e1) {  // receiver done (or empty): move to the next one");
        S.ind++;
        S("r += G;");
        S("if (r >= N) break;");
        S("eb = nb; e1 = n1;");
        if (R.gst) S("fresh = true;");
        S("if (r + G < N) { nb = " + off_at(R, "r + G") + "; n1 = " + off_at(R, "r + G + 1") + "; }");
        for (int j = 0; j < CH; ++j) S(fmt("sv%d = (%d < e1 - eb) ? %s : 0;", j, j, src_at(R, fmt("eb + %d", j)).c_str()));
        S("continue;");
        S.ind--;
        S("}");
        S(fmt("const int ne = min(%s_CH, e1 - eb);", pre));
        S(fmt("const int ebn = eb + %s_CH;", pre));
        for (int j = 0; j < CH; ++j)
            S(fmt("const int svn%d = (ebn + %d < e1) ? %s : 0;", j, j, src_at(R, fmt("ebn + %d", j)).c_str()));
        if (R.pf > 0) {
            // L2 prefetch of the w (and Y) rows R.pf chunks ahead, in this receiver or the next
            S(fmt("{ int pa = eb + %d, pb; bool ok = true;", R.pf * CH));
            S(fmt("  if (pa < e1) { pb = min(pa + %s_CH, e1); }", pre));
            S(fmt("  else if (r + G < N) { pa = nb + (pa - e1); pb = min(pa + %s_CH, n1); ok = pa < n1; }", pre));
            S("  else { ok = false; pb = pa; }");
            S(fmt("  if (ok) { prefetch_l2(w + (size_t)pa * (UVU_P * UVU_U), (unsigned)(pb - pa) * %zuu);", wbytes()));
            if (R.ybulk) S(fmt("             prefetch_l2(Y + (size_t)pa * UVU_DY, (unsigned)(pb - pa) * %zuu); }", ybytes()));
            else S("  }");
            S("}");
        }
        if (R.gst) {
            // first chunk of a receiver: its d_out block goes into the (single) block buffer once
            // the consumers have taken the previous receiver's block into registers
            S("if (fresh) {");
            S(fmt("  if (kg >= 1u && !mbar_wait(sbase + %s_GBAR + 8u, (kg - 1u) & 1u)) { dead = true; break; }", pre));
            S(fmt("  mbar_expect_tx(sbase + %s_GBAR, %zuu);", pre, R.gbytes));
            S(fmt("  bulk_g2s(sbase + %s_GBUF, gout + (size_t)r * (UVU_U * UVU_DO), %zuu, sbase + %s_GBAR);", pre, R.gbytes, pre));
            S("  ++kg;");
            S("  fresh = false;");
            S("}");
        }
        S(fmt("const unsigned st = c %% %s_NST;", pre));
        S(fmt("if (c >= %s_NST && !mbar_wait(sbase + %s_BAR + 8u * (%s_NST + st), ((c / %s_NST) - 1u) & 1u)) { dead = true; break; }",
              pre, pre, pre, pre));
        S(fmt("const unsigned full = sbase + %s_BAR + 8u * st;", pre));
        S(fmt("const unsigned stg = sbase + st * %s_STAGE;", pre));
        if (R.dual) S("mbar_expect_tx(full, (unsigned)ne * txe);");
        else S(fmt("mbar_expect_tx(full, (unsigned)ne * %s_TX);", pre));
        if (!R.wsh) S(fmt("bulk_g2s(stg, w + (size_t)eb * (UVU_P * UVU_U), (unsigned)ne * %zuu, full);", wbytes()));
        if (R.dual) S(fmt("if (hm & 4) bulk_g2s(stg + %s_AWOFF, aw + (size_t)eb * (UVU_P * UVU_U), (unsigned)ne * %zuu, full);", pre, wbytes()));
        if (R.ybulk) S(fmt("bulk_g2s(stg + %s_YOFF, Y + (size_t)eb * UVU_DY, (unsigned)ne * %zuu, full);", pre, ybytes()));
        if (R.ybulk && R.dual) S(fmt("if (hm & 2) bulk_g2s(stg + %s_AYOFF, aY + (size_t)eb * UVU_DY, (unsigned)ne * %zuu, full);", pre, ybytes()));
        if (R.xbulk) {
            for (int j = 0; j < CH; ++j)
                S(fmt("if (%d < ne) bulk_g2s(stg + %s_XOFF + %zuu, x + (size_t)sv%d * (UVU_U * UVU_DX), %zuu, full);", j, pre,
                      size_t(j) * xbytes(), j, xbytes()));
            if (R.dual)
                for (int j = 0; j < CH; ++j)
                    S(fmt("if ((hm & 1) && %d < ne) bulk_g2s(stg + %s_AXOFF + %zuu, ax + (size_t)sv%d * (UVU_U * UVU_DX), %zuu, full);",
                          j, pre, size_t(j) * xbytes(), j, xbytes()));
        }
        for (int j = 0; j < CH; ++j) S(fmt("sv%d = svn%d;", j, j));
        S("eb = ebn;");
        S("++c;");
        S.ind--;
        S("}");
        S("if (dead) {  // let the copies already issued land before the block exits");
        S(fmt("  const unsigned n = c < %s_NST ? c : %s_NST;", pre, pre));
        S(fmt("  for (unsigned k = c - n; k < c; ++k) mbar_wait(sbase + %s_BAR + 8u * (k %% %s_NST), (k / %s_NST) & 1u);", pre, pre, pre));
        if (R.gst) S(fmt("  if (kg >= 1u) mbar_wait(sbase + %s_GBAR, (kg - 1u) & 1u);", pre));
        S("}");
        S.ind--;
        S("}");
    }

    // Operand loads of edge slot j of a stage for the receiver kernels.
    void emit_stage_edge_loads(Src& S, const RecvPipe& R, const char* pre, const std::set<int>& xn,
                               const std::set<int>& yn, const std::vector<int>& paths) const {
        S("const int e = eb + j;");
        if (R.xbulk) {
            emit_row_loads(S, "xv", fmt("reinterpret_cast<const %s*>(stg + %s_XOFF) + (j * UVU_U + u) * UVU_DX", T.c_str(), pre),
                           P->Dx, xn, false);
        } else {
            S("const int s = " + src_at(R, "e") + ";");
            emit_row_loads(S, "xv", "x + ((size_t)s * UVU_U + u) * UVU_DX", P->Dx, xn);
        }
        if (R.ybulk)
            emit_row_loads(S, "yv", fmt("reinterpret_cast<const %s*>(stg + %s_YOFF) + j * UVU_DY", T.c_str(), pre), P->Dy, yn,
                           false);
        else
            emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        if (R.wsh) {  // batch-shared weights: the channel's row, cached by L1 across samples
            for (int pi : paths) S(fmt("const %s wv_%d = __ldg(w + %d * UVU_U + u);", T.c_str(), pi, pi));
        } else {
            S(fmt("const %s* swr = reinterpret_cast<const %s*>(stg) + j * (UVU_P * UVU_U) + u;", T.c_str(), T.c_str()));
            for (int pi : paths) S(fmt("const %s wv_%d = swr[%d * UVU_U];", T.c_str(), pi, pi));
        }
        if (!R.dual) return;
        // cotangent rows of the double backward; absent ones (mask hm) read as zero
        if (R.xbulk) {
            emit_row_loads_masked(S, "axv", fmt("reinterpret_cast<const %s*>(stg + %s_AXOFF) + (j * UVU_U + u) * UVU_DX", T.c_str(), pre),
                                  P->Dx, xn, "hm & 1", false);
        } else {
            emit_row_loads_masked(S, "axv", "ax + ((size_t)s * UVU_U + u) * UVU_DX", P->Dx, xn, "hm & 1");
        }
        if (R.ybulk)
            emit_row_loads_masked(S, "ayv", fmt("reinterpret_cast<const %s*>(stg + %s_AYOFF) + j * UVU_DY", T.c_str(), pre), P->Dy, yn,
                                  "hm & 2", false);
        else
            emit_row_loads_masked(S, "ayv", "aY + (size_t)e * UVU_DY", P->Dy, yn, "hm & 2");
        for (int pi : paths) S(fmt("%s awv_%d = 0;", T.c_str(), pi));
        S("if (hm & 4) {");
        S(fmt("  const %s* swa = reinterpret_cast<const %s*>(stg + %s_AWOFF) + j * (UVU_P * UVU_U) + u;", T.c_str(), T.c_str(), pre));
        for (int pi : paths) S(fmt("  awv_%d = swa[%d * UVU_U];", pi, pi));
        S("}");
    }

    void emit_fwd_v2(Src& S, const RecvPipe& R) const {
        const int NG = int(P->groups.size());
        emit_recv_producer(S, R, "FW", "fwd_producer");
        // The receiver's out row accumulates in column-scaled form (acc_k = out_k / s_k), written
        // back scaled once per receiver: fp64 plans (bound by the FP64 pipe; 49.6 -> 37.7 ms) and
        // fp32 plans with out rows of at most 64 values (MACE-medium 0.340 -> 0.329 ms; its
        // double-backward forward 0.835 -> 0.797 ms with 8 bytes of spill).  ptxas gave the wider
        // fp32 forwards (MACE-large, wide) more registers or spills in the scaled form, so they
        // keep the unscaled one.
        const std::vector<double> scales = column_scales();
        colscale = ((f64 || P->Do <= 64) && !R.tp && col_scale_enabled()) ? &scales : nullptr;
        for (int g = 0; g < NG; ++g) {
            const std::vector<int>& paths = P->groups[g];
            const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
            std::vector<int> outs;
            for (int pi : paths)
                for (int m = 0; m < 2 * P->paths[pi].l3 + 1; ++m) outs.push_back(P->paths[pi].ooff + m);
            S(fmt("__device__ __forceinline__ void fwd_rcv%d(int e0, int e1, int u, bool uvalid, int lane, unsigned& c, bool& dead,", g));
            S(fmt("    const unsigned char* smem, unsigned sbase, const int* __restrict__ src, const %s* __restrict__ x,", T.c_str()));
            if (R.dual) S(fmt("    const %s* __restrict__ ax, const %s* __restrict__ aY, int hm,", T.c_str(), T.c_str()));
            S(fmt("    const %s* __restrict__ Y, const %s* __restrict__ w, %s* __restrict__ orow) {", T.c_str(), T.c_str(), T.c_str()));
            S.ind++;
            for (int k : outs) S(fmt("%s acc_%d = 0;", T.c_str(), k));
            S("for (int eb = e0; eb < e1; eb += FW_CH, ++c) {");
            S.ind++;
            S("const unsigned st = c % FW_NST;");
            S("if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(sbase + FW_BAR + 8u * st, (c / FW_NST) & 1u));");
            S("if (dead) continue;");
            S("const int ne = min(FW_CH, e1 - eb);");
            S("const unsigned char* stg = smem + st * FW_STAGE;");
            S("if (uvalid) {");
            S.ind++;
            S("#pragma unroll");
            S("for (int j = 0; j < FW_CH; ++j) {");
            S.ind++;
            S("if (j < ne) {");
            S.ind++;
            emit_stage_edge_loads(S, R, "FW", xn, yn, paths);
            if (R.dual) emit_hvp_fwd_edge(S, paths);
            else emit_fwd_edge(S, paths);
            S.ind--;
            S("}");
            S.ind--;
            S("}");
            S.ind--;
            S("}");
            emit_release(S, "FW");
            S.ind--;
            S("}");
            S("if (uvalid) {");
            for (int k : outs) S(fmt("  orow[%d] = %s;", k, gload(k, fmt("acc_%d", k)).c_str()));
            S("}");
            S.ind--;
            S("}");
        }
        colscale = nullptr;
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_NCT + 32, FW_MINB) %s(long long N, const int* __restrict__ off,",
              R.dual ? "uvu_hvp_fwd" : R.tp ? (R.wsh ? "uvu_tp_fwd_sh" : "uvu_tp_fwd") : "uvu_fwd"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y,", T.c_str(), T.c_str()));
        if (R.dual)
            S(fmt("    const %s* __restrict__ w, const %s* __restrict__ ax, const %s* __restrict__ aY, const %s* __restrict__ aw, int hm,",
                  T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        else
            S(fmt("    const %s* __restrict__ w,", T.c_str()));
        S(fmt("    %s* __restrict__ out) {", T.c_str()));
        S.ind++;
        S("extern __shared__ __align__(128) unsigned char smem[];");
        S("const unsigned sbase = smem_addr(smem);");
        S("const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;");
        S("if (tid == 0) {");
        S("  for (int i = 0; i < FW_NST; ++i) { mbar_init(sbase + FW_BAR + 8u * i, 1u); mbar_init(sbase + FW_BAR + 8u * (FW_NST + i), " + std::string(empty_count("UVU_NCW", "UVU_NCT")) + "); }");
        S("  asm volatile(\"fence.mbarrier_init.release.cluster;\" ::: \"memory\");");
        S("}");
        S("__syncthreads();");
        S("if (warp == UVU_NCW) {");
        if (R.dual) S("  if (lane == 0) fwd_producer(N, off, src, x, Y, w, nullptr, ax, aY, aw, hm, sbase);");
        else S("  if (lane == 0) fwd_producer(N, off, src, x, Y, w, nullptr, sbase);");
        S("  return;");
        S("}");
        S("const int u = tid % UVU_UP, g = tid / UVU_UP;");
        S("const bool uvalid = u < UVU_U;");
        S("unsigned c = 0;");
        S("bool dead = false;");
        if (R.odp == 0) {
            S("for (long long r = blockIdx.x; r < N; r += gridDim.x) {");
            S.ind++;
            S("const int e0 = " + off_at(R, "r") + ", e1 = " + off_at(R, "r + 1") + ";");
            S(T + "* orow = out + ((size_t)r * UVU_U + u) * UVU_DO;");
            for (int g = 0; g < NG; ++g)
                S(fmt("%sif (g == %d) fwd_rcv%d(e0, e1, u, uvalid, lane, c, dead, smem, sbase, src, x, %sY, w, orow);", g ? "else " : "", g, g,
                      R.dual ? "ax, aY, hm, " : ""));
            S.ind--;
            S("}");
            S.ind--;
            S("}");
            return;
        }
        S(fmt("%s* const sout = reinterpret_cast<%s*>(smem + FW_OBUF);", T.c_str(), T.c_str()));
        S(fmt("%s* const orow = sout + u * FW_ODP;", T.c_str()));
        if (R.ovec) S("const bool ovec = (reinterpret_cast<size_t>(out) & 15) == 0;");
        S("for (long long r = blockIdx.x; r < N; r += gridDim.x) {");
        S.ind++;
        S("const int e0 = " + off_at(R, "r") + ", e1 = " + off_at(R, "r + 1") + ";");
        S("consumer_sync();  // the previous receiver's block has been copied out of sout");
        for (int g = 0; g < NG; ++g)
            S(fmt("%sif (g == %d) fwd_rcv%d(e0, e1, u, uvalid, lane, c, dead, smem, sbase, src, x, %sY, w, orow);", g ? "else " : "", g, g,
                  R.dual ? "ax, aY, hm, " : ""));
        S("consumer_sync();");
        S(fmt("%s* const og = out + (size_t)r * (UVU_U * UVU_DO);", T.c_str()));
        if (R.ovec) {
            const int nv = int(size_t(P->U) * P->Do * P->elem() / 16);
            S("if (ovec) {");
            S(fmt("  for (int i = tid; i < %d; i += UVU_NCT) reinterpret_cast<float4*>(og)[i] = reinterpret_cast<const float4*>(sout)[i];", nv));
            S("} else {");
            S("  for (int i = tid; i < UVU_U * UVU_DO; i += UVU_NCT) og[i] = sout[i];");
            S("}");
        } else if (R.odp == P->Do) {
            S("for (int i = tid; i < UVU_U * UVU_DO; i += UVU_NCT) og[i] = sout[i];");
        } else {
            S("for (int i = tid; i < UVU_U * UVU_DO; i += UVU_NCT) {");
            S("  const int uu = i / UVU_DO;");
            S("  og[i] = sout[uu * FW_ODP + (i - uu * UVU_DO)];");
            S("}");
        }
        S.ind--;
        S("}");
        S.ind--;
        S("}");
    }

    // Warp transpose-reduction of the dY partials of one edge over the 32 channels of the warp,
    // then one lane per component stores the warp sum into the stage's partial buffer.
    // Values are halved level by level (each lane keeps one half and receives the other half of
    // its xor partner), so D values over 32 lanes take about D shuffles instead of 5 D.
    // dY's sum over the warp's 32 channels through a shared-memory tile: lane l writes its D
    // (<= 16) values as row l (four 16-byte stores, the 16-byte groups rotated by (l >> 1) & 3 so
    // that each quarter-warp's stores hit 32 distinct banks), then lane l sums column l & 15 over
    // the rows of its half-warp in ascending order (16 loads, conflict-free: the halves' rows
    // start in opposite bank halves) and the two halves are added by one shuffle.  The order of
    // the additions is fixed, so dY stays bitwise repeatable.
    void emit_dy_tile_reduce(Src& S, const std::vector<int>& K, const char* pre) const {
        const int D = int(K.size());
        S("{");
        S.ind++;
        S(fmt("float* const dyt = reinterpret_cast<float*>(const_cast<unsigned char*>(smem) + %s_DYT) + warp * %d;", pre, kDytWords));
        S("float4* const trow = reinterpret_cast<float4*>(dyt + lane * 16 + ((lane & 16) ? 16 : 0));");
        S("const int tsw = (lane >> 1) & 3;");
        for (int c = 0; c < 4; ++c) {
            std::string v[4];
            for (int i = 0; i < 4; ++i) v[i] = (4 * c + i < D) ? fmt("dyp_%d", K[4 * c + i]) : "0.0f";
            S(fmt("trow[%d ^ tsw] = make_float4(%s, %s, %s, %s);", c, v[0].c_str(), v[1].c_str(), v[2].c_str(), v[3].c_str()));
        }
        S("__syncwarp();");
        S("const int tm = lane & 15, tg = tm >> 2;");
        S("const float* const tcol = dyt + ((lane & 16) ? 272 : 0) + (tm & 3);");
        S("const int to0 = (tg ^ 0) << 2, to1 = (tg ^ 1) << 2, to2 = (tg ^ 2) << 2, to3 = (tg ^ 3) << 2;");
        for (int r = 0; r < 16; ++r) {
            const int c = (r >> 1) & 3;
            if (r == 0) S(fmt("float ts = tcol[%d + to%d];", r * 16, c));
            else S(fmt("ts += tcol[%d + to%d];", r * 16, c));
        }
        S("ts += __shfl_xor_sync(0xffffffffu, ts, 16);");
        S("__syncwarp();");
        bool contiguous = true;
        for (int i = 1; i < D; ++i) contiguous = contiguous && K[i] == K[0] + i;
        std::string comp;
        if (contiguous) {
            comp = fmt("%d + tm", K[0]);
        } else {
            comp = "-1";
            for (int i = D - 1; i >= 0; --i) comp = fmt("(tm == %d ? %d : %s)", i, K[i], comp.c_str());
        }
        S(fmt("if (lane < %d) part[j * UVU_DY + (%s)] = ts;", D, comp.c_str()));
        std::set<int> ks(K.begin(), K.end());
        for (int k = 0; k < P->Dy; ++k)
            if (!ks.count(k)) S(fmt("if (lane == 0) part[j * UVU_DY + %d] = 0;", k));
        S.ind--;
        S("}");
    }

    void emit_dy_warp_reduce(Src& S, const std::vector<int>& K) const {
        const int D = int(K.size());
        int P2 = 1;
        while (P2 < D) P2 *= 2;
        std::vector<std::string> v(P2);
        for (int i = 0; i < P2; ++i) {
            v[i] = fmt("rv_%d", i);
            S(fmt("%s %s = %s;", T.c_str(), v[i].c_str(), i < D ? fmt("dyp_%d", K[i]).c_str() : "0"));
        }
        int len = P2;
        int idx_terms_off[5], idx_terms_half[5], nsplit = 0, lowmask = 0;
        for (int o = 16; o >= 1; o >>= 1) {
            if (len > 1) {
                const int h = len / 2;
                S(fmt("{ const bool hi = (lane & %d) != 0;", o));
                for (int i = 0; i < h; ++i) {
                    S(fmt("  const %s snd_%d = hi ? %s : %s;", T.c_str(), i, v[i].c_str(), v[i + h].c_str()));
                    S(fmt("  const %s kep_%d = hi ? %s : %s;", T.c_str(), i, v[i + h].c_str(), v[i].c_str()));
                }
                for (int i = 0; i < h; ++i)
                    S(fmt("  %s = kep_%d + __shfl_xor_sync(0xffffffffu, snd_%d, %d);", v[i].c_str(), i, i, o));
                S("}");
                idx_terms_off[nsplit] = o;
                idx_terms_half[nsplit] = h;
                ++nsplit;
                len = h;
            } else {
                S(fmt("%s += __shfl_xor_sync(0xffffffffu, %s, %d);", v[0].c_str(), v[0].c_str(), o));
                lowmask |= o;
            }
        }
        std::string idx = "0";
        for (int i = 0; i < nsplit; ++i)
            idx += fmt(" + ((lane & %d) ? %d : 0)", idx_terms_off[i], idx_terms_half[i]);
        S(fmt("{ const int idx = %s;", idx.c_str()));
        bool contiguous = true;
        for (int i = 1; i < D; ++i) contiguous = contiguous && K[i] == K[0] + i;
        std::string comp;
        if (contiguous) {
            comp = fmt("%d + idx", K[0]);
        } else {
            comp = "-1";
            for (int i = D - 1; i >= 0; --i) comp = fmt("(idx == %d ? %d : %s)", i, K[i], comp.c_str());
        }
        S(fmt("  if ((lane & %d) == 0 && idx < %d) part[j * UVU_DY + (%s)] = %s; }", lowmask, D, comp.c_str(), v[0].c_str()));
        std::set<int> ks(K.begin(), K.end());
        for (int k = 0; k < P->Dy; ++k)
            if (!ks.count(k)) S(fmt("if (lane == 0) part[j * UVU_DY + %d] = 0;", k));
    }

    void emit_edge_v2(Src& S, const RecvPipe& R) const {
        const int NG = int(P->groups.size());
        dw_accum = R.wsh;
        emit_recv_producer(S, R, "EG", "edge_producer");
        // d_out rows held in registers for the receiver's edges take column scales
        const std::vector<double> scales = column_scales();
        colscale = (!R.tp && col_scale_enabled() && (!R.gsm || R.gst)) ? &scales : nullptr;
        obulk = edge_bulk_out_enabled() && R.ch == 1 && !R.dual && !R.tp && !R.wsh && !R.lastwarp && NG == 1 &&
                R.xbulk && wbytes() % 16 == 0 && release_mode() != 1;
        for (int g = 0; g < NG; ++g) {
            const std::vector<int>& paths = P->groups[g];
            const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
            std::vector<int> outs;
            for (int pi : paths)
                for (int m = 0; m < 2 * P->paths[pi].l3 + 1; ++m) outs.push_back(P->paths[pi].ooff + m);
            S(fmt("__device__ __forceinline__ void edge_rcv%d(long long r, int e0, int e1, int u, bool uvalid, int lane, int warp,", g));
            S("    int tid, unsigned& c, unsigned& kg, bool& dead, int& buf, const unsigned char* smem, unsigned sbase,");
            S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y,", T.c_str(), T.c_str()));
            if (R.dual) S(fmt("    const %s* __restrict__ ax, const %s* __restrict__ aY, int hm,", T.c_str(), T.c_str()));
            S(fmt("    const %s* __restrict__ gout, %s* __restrict__ dY, %s* __restrict__ dw, %s* __restrict__ dx,",
                  T.c_str(), T.c_str(), T.c_str(), T.c_str()));
            std::string dwa;
            if (R.wsh)
                for (int pi : paths) dwa += fmt(", %s& dwa_%d", T.c_str(), pi);
            S(fmt("    %s* __restrict__ dxe, int g, const %s* __restrict__ w%s) {", T.c_str(), T.c_str(), dwa.c_str()));
            S.ind++;
            if (R.gst && R.gsm) {
                // d_out row of this channel read from the receiver's staged block at each use
                S(fmt("const %s* grow = reinterpret_cast<const %s*>(smem + EG_GBUF) + (uvalid ? u : 0) * UVU_DO;", T.c_str(), T.c_str()));
                S("if (e1 > e0 && !dead) dead = !__all_sync(0xffffffffu, mbar_wait(sbase + EG_GBAR, kg & 1u));");
                if (colscale) {
                    // the thread's own row of the block, scaled in place once per receiver (the
                    // consumers hold the block until the receiver is done)
                    S("if (e1 > e0 && !dead && uvalid) {");
                    S.ind++;
                    S(fmt("%s* gw = const_cast<%s*>(grow);", T.c_str(), T.c_str()));
                    for (int k : outs)
                        if (cs(k) != 1.0) S(fmt("gw[%d] = %s;", k, gload(k, fmt("gw[%d]", k)).c_str()));
                    S.ind--;
                    S("}");
                }
            } else if (R.gst) {
                // d_out row of this channel from the receiver's staged block; the block buffer
                // is handed back to the producer as soon as the row is in registers
                for (int k : outs) S(fmt("%s gv_%d = 0;", T.c_str(), k));
                S("if (e1 > e0) {");
                S.ind++;
                S("if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(sbase + EG_GBAR, kg & 1u));");
                S(fmt("const %s* grow = reinterpret_cast<const %s*>(smem + EG_GBUF) + (uvalid ? u : 0) * UVU_DO;", T.c_str(), T.c_str()));
                for (int k : outs) S(fmt("gv_%d = %s;", k, gload(k, fmt("grow[%d]", k)).c_str()));
                S("if (!dead) {");
                S.ind++;
                if (release_mode() != 3) S("__threadfence_block();");
                S("asm volatile(\"fence.proxy.async.shared::cta;\" ::: \"memory\");");
                S("__syncwarp();");
                S(std::string("if (") + (release_mode() == 1 ? "true" : "lane == 0") + ") mbar_arrive(sbase + EG_GBAR + 8u);");
                S.ind--;
                S("}");
                S("++kg;");
                S.ind--;
                S("}");
            } else {
                S(fmt("const %s* __restrict__ grow = gout + ((size_t)r * UVU_U + (uvalid ? u : 0)) * UVU_DO;", T.c_str()));
                for (int k : outs) S(fmt("const %s gv_%d = %s;", T.c_str(), k, gload(k, fmt("__ldg(grow + %d)", k)).c_str()));
            }
            S(fmt("%s* partbase = reinterpret_cast<%s*>(const_cast<unsigned char*>(smem) + EG_PART);", T.c_str(), T.c_str()));
            S("for (int eb = e0; eb < e1; eb += EG_CH, ++c) {");
            S.ind++;
            S("const unsigned st = c % EG_NST;");
            S("if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(sbase + EG_BAR + 8u * st, (c / EG_NST) & 1u));");
            S("const int ne = min(EG_CH, e1 - eb);");
            S("const unsigned char* stg = smem + st * EG_STAGE;");
            S(fmt("%s* part = partbase + (size_t)(buf * UVU_NCW + warp) * EG_CH * UVU_DY;", T.c_str()));
            S("if (!dead) {");
            S.ind++;
            S("#pragma unroll");
            S("for (int j = 0; j < EG_CH; ++j) {");
            S.ind++;
            S("if (j < ne) {");
            S.ind++;
            for (int k : yn) S(fmt("%s dyp_%d = 0;", T.c_str(), k));
            S("if (uvalid) {");
            S.ind++;
            emit_stage_edge_loads(S, R, "EG", xn, yn, paths);
            if (obulk)  // dw goes where this thread read its w values, then out with the stage
                S(fmt("%s* dwe = reinterpret_cast<%s*>(const_cast<unsigned char*>(stg)) + j * (UVU_P * UVU_U) + u;", T.c_str(), T.c_str()));
            else if (!R.wsh)
                S(T + "* __restrict__ dwe = dw + (size_t)e * (UVU_P * UVU_U) + u;");
            for (int k : xn) S(fmt("%s dxp_%d = 0;", T.c_str(), k));
            // staged-row kernels pair only dY's contraction (the full pairing spilled there);
            // measured: MACE-large VJP 2.560 -> 2.515 ms, wide 5.287 -> 5.185 ms.  So do the
            // double-backward kernels with rows of at most 64 values, in both of their contractions
            // (MACE-medium 1.487 -> 1.454 ms); with wider rows (MACE-large, wide) it added spills.
            pair_dy_only = R.gsm || R.dual;
            pair_contract = colscale && !(R.dual && (R.gsm || P->Do > 64)) && pack_products() && pair_contract_enabled();
            if (pair_contract && !pair_dy_only)
                for (int k : xn) {
                    S(fmt("const unsigned long long xb_%d = uvu_f2pack(xv_%d, xv_%d);", k, k, k));
                    S(fmt("unsigned long long dxq_%d = 0ull;", k));
                }
            // pair loads need every row of the staged block to start 8-byte (fp64: 16-byte)
            // aligned: an even D_out (the block itself starts 16-byte aligned)
            const bool gq = R.gsm && !R.dual && P->Do % 2 == 0 && R.g_off % 16 == 0 && gsm_vec_enabled();
            id_fold = !R.dual && id_fold_enabled();
            auto gval = [&R, gq](int k) { return R.gsm ? (gq ? fmt("gq_%d", k) : fmt("grow[%d]", k)) : fmt("gv_%d", k); };
            if (R.dual) {
                // dw(x<-ax) + dw(Y<-aY) through the mixed products; dY(x<-ax) and dx(Y<-aY) with
                // w; dY and dx with w<-aw
                S("if (dw) {");
                S.ind++;
                emit_mixed_products(S, paths, "q");
                emit_bwd_pairs(S, paths, true, false, false, gval);
                S.ind--;
                S("}");
                emit_bwd_pairs(S, paths, false, true, true, gval, "axv", "ayv", "wv");
                emit_bwd_pairs(S, paths, false, true, true, gval, "xv", "yv", "awv");
            } else if (R.gsm) {
                // one pass per (x irrep, SH irrep) pair: its products, then per path dw, a = w g and
                // h, then the pair's dY / dx contraction, so each d_out value is read and used within
                // its path's block
                local_products = true;
                guard_dw = true;
                gsm_vec = gq;
                emit_bwd_pairs(S, paths, true, true, true, gval);
                gsm_vec = false;
                local_products = false;
                guard_dw = false;
            } else {
                emit_products(S, paths);
                if (id_fold)  // the identity paths' zi serve dw and the dY / dx below
                    for (int pi : paths)
                        if (is_identity(P->paths[pi])) {
                            emit_identity_z(S, pi, gval);
                            zi_ready.insert(pi);
                        }
                S("if (dw) {");
                S.ind++;
                emit_bwd_pairs(S, paths, true, false, false, gval);
                S.ind--;
                S("}");
                emit_bwd_pairs(S, paths, false, true, true, gval);
                zi_ready.clear();
            }
            if (pair_contract && !pair_dy_only)
                for (int k : xn) S(fmt("{ float lo, hi; uvu_f2unpack(dxq_%d, lo, hi); dxp_%d += lo + hi; }", k, k));
            pair_contract = pair_dy_only = false;
            S("if (dx) {");
            S.ind++;
            if (!R.xbulk) {
                S(T + "* __restrict__ dxr = dx + ((size_t)s * UVU_U + u) * UVU_DX;");
            } else {
                S("const int s = " + src_at(R, "e") + ";");
                S(T + "* __restrict__ dxr = dx + ((size_t)s * UVU_U + u) * UVU_DX;");
            }
            emit_dx_atomics(S, xn);
            S.ind--;
            S("}");
            emit_dx_edge_store(S, xn, NG);
            S.ind--;
            S("}");  // uvalid
            S("if (dY) {");
            S.ind++;
            std::vector<int> K(yn.begin(), yn.end());
            if (R.dyt && K.size() > 8) emit_dy_tile_reduce(S, K, "EG");
            else emit_dy_warp_reduce(S, K);
            S.ind--;
            S("}");
            S.ind--;
            S("}");  // j < ne
            S.ind--;
            S("}");  // j
            if (obulk) {  // the stage goes back to the producer after its outputs have left it
                if (release_mode() != 3) S("__threadfence_block();");
                S("asm volatile(\"fence.proxy.async.shared::cta;\" ::: \"memory\");");
            } else {
                emit_release(S, "EG");
            }
            S.ind--;
            S("}");  // !dead
            if (R.lastwarp) {
                // the last warp to finish the stage sums the warps' dY partials; the others go on
                S("if (!dead && dY) {");
                S.ind++;
                S("unsigned* const cnt = reinterpret_cast<unsigned*>(const_cast<unsigned char*>(smem) + EG_CNT);");
                S("__syncwarp();");
                S("unsigned last = 0;");
                S("if (lane == 0) { __threadfence_block(); last = atomicAdd(cnt + buf, 1u) == UVU_NCW - 1; }");
                S("last = __shfl_sync(0xffffffffu, last, 0);");
                S("if (last) {");
                S.ind++;
                S("__threadfence_block();");
                S("for (int t = lane; t < ne * UVU_DY; t += 32) {");
                S.ind++;
                S("const int j = t / UVU_DY, k = t - j * UVU_DY;");
                S(T + " acc = 0;");
                S("#pragma unroll");
                S("for (int wp = 0; wp < UVU_NCW; ++wp) acc += partbase[((size_t)(buf * UVU_NCW + wp) * EG_CH + j) * UVU_DY + k];");
                S("dY[(size_t)(eb + j) * UVU_DY + k] = acc;");
                S.ind--;
                S("}");
                S("__syncwarp();");
                S("if (lane == 0) cnt[buf] = 0u;");
                S.ind--;
                S("}");
                S.ind--;
                S("}");
                S("buf = buf == EG_NBUF - 1 ? 0 : buf + 1;");
                S.ind--;
                S("}");
                S.ind--;
                S("}");
            } else {
            S("consumer_sync();");
            if (obulk) {
                S("if (tid == 0 && !dead) {");
                S.ind++;
                S("const unsigned sst = sbase + st * EG_STAGE;");
                S(fmt("if (dw) bulk_s2g(dw + (size_t)eb * (UVU_P * UVU_U), sst, (unsigned)ne * %zuu);", wbytes()));
                S(fmt("if (dxe) bulk_s2g(dxe + (size_t)eb * (UVU_U * UVU_DX), sst + EG_XOFF, (unsigned)ne * %zuu);", xbytes()));
                S("bulk_commit();");
                S("bulk_wait_read();");
                S("mbar_arrive(sbase + EG_BAR + 8u * (EG_NST + st));");
                S.ind--;
                S("}");
            }
            if (NG > 1) {
                S("if (!dead && dxe) {");
                S.ind++;
                S(fmt("const %s* xpb = reinterpret_cast<const %s*>(smem + EG_XPART) + (size_t)buf * (UVU_G * EG_CH * UVU_UP * UVU_DX);", T.c_str(), T.c_str()));
                S("for (int t = tid; t < ne * UVU_UP * UVU_DX; t += UVU_NCT) {");
                S.ind++;
                S("const int k = t % UVU_DX, uu = (t / UVU_DX) % UVU_UP, j = t / (UVU_DX * UVU_UP);");
                S("if (uu < UVU_U) {");
                S.ind++;
                S(T + " acc = 0;");
                S("#pragma unroll");
                S("for (int gg = 0; gg < UVU_G; ++gg) acc += xpb[((size_t)(gg * EG_CH + j) * UVU_UP + uu) * UVU_DX + k];");
                S("dxe[((size_t)(eb + j) * UVU_U + uu) * UVU_DX + k] = acc;");
                S.ind--;
                S("}");
                S.ind--;
                S("}");
                S.ind--;
                S("}");
            }
            S("if (!dead && dY) {");
            S.ind++;
            S("for (int t = tid; t < ne * UVU_DY; t += UVU_NCT) {");
            S.ind++;
            S("const int j = t / UVU_DY, k = t - j * UVU_DY;");
            S(T + " acc = 0;");
            S("#pragma unroll");
            S("for (int wp = 0; wp < UVU_NCW; ++wp) acc += partbase[((size_t)(buf * UVU_NCW + wp) * EG_CH + j) * UVU_DY + k];");
            S("dY[(size_t)(eb + j) * UVU_DY + k] = acc;");
            S.ind--;
            S("}");
            S.ind--;
            S("}");
            S("buf ^= 1;");
            S.ind--;
            S("}");
            if (R.gst && R.gsm) {  // the receiver is done: its d_out block goes back to the producer
                S("if (e1 > e0) {");
                S.ind++;
                S("if (!dead) {");
                S.ind++;
                if (release_mode() != 3) S("__threadfence_block();");
                S("asm volatile(\"fence.proxy.async.shared::cta;\" ::: \"memory\");");
                S("__syncwarp();");
                S(std::string("if (") + (release_mode() == 1 ? "true" : "lane == 0") + ") mbar_arrive(sbase + EG_GBAR + 8u);");
                S.ind--;
                S("}");
                S("++kg;");
                S.ind--;
                S("}");
            }
            S.ind--;
            S("}");
            }
        }
        colscale = nullptr;
        id_fold = false;
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_NCT + 32, EG_MINB) %s(long long N, const int* __restrict__ off,",
              R.dual ? "uvu_hvp_edge" : R.tp ? (R.wsh ? "uvu_tp_edge_sh" : "uvu_tp_edge") : "uvu_bwd_edge"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y,", T.c_str(), T.c_str()));
        if (R.dual)
            S(fmt("    const %s* __restrict__ w, const %s* __restrict__ gout, const %s* __restrict__ ax, const %s* __restrict__ aY,\n"
                  "    const %s* __restrict__ aw, int hm, %s* __restrict__ dY, %s* __restrict__ dw,",
                  T.c_str(), T.c_str(), T.c_str(), T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        else
            S(fmt("    const %s* __restrict__ w, const %s* __restrict__ gout, %s* __restrict__ dY, %s* __restrict__ dw,",
                  T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    %s* __restrict__ dx, %s* __restrict__ dxe) {", T.c_str(), T.c_str()));
        S.ind++;
        S("extern __shared__ __align__(128) unsigned char smem[];");
        S("const unsigned sbase = smem_addr(smem);");
        S("const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;");
        S("if (tid == 0) {");
        S("  for (int i = 0; i < EG_NST; ++i) { mbar_init(sbase + EG_BAR + 8u * i, 1u); mbar_init(sbase + EG_BAR + 8u * (EG_NST + i), " + std::string(obulk ? "1u" : empty_count("UVU_NCW", "UVU_NCT")) + "); }");
        if (R.gst) S("  mbar_init(sbase + EG_GBAR, 1u); mbar_init(sbase + EG_GBAR + 8u, " + std::string(empty_count("UVU_NCW", "UVU_NCT")) + ");");
        if (R.lastwarp) S("  for (int i = 0; i < EG_NBUF; ++i) reinterpret_cast<unsigned*>(smem + EG_CNT)[i] = 0u;");
        S("  asm volatile(\"fence.mbarrier_init.release.cluster;\" ::: \"memory\");");
        S("}");
        S("__syncthreads();");
        S("if (warp == UVU_NCW) {");
        if (R.dual) S("  if (lane == 0) edge_producer(N, off, src, x, Y, w, gout, ax, aY, aw, hm, sbase);");
        else S("  if (lane == 0) edge_producer(N, off, src, x, Y, w, gout, sbase);");
        S("  return;");
        S("}");
        S("const int u = tid % UVU_UP, g = tid / UVU_UP;");
        S("const bool uvalid = u < UVU_U;");
        S("unsigned c = 0, kg = 0;");
        S("bool dead = false;");
        S("int buf = 0;");
        // dw of batch-shared weights: this block's sum over its samples, per thread.  An fp32 plan
        // sums 16 samples in registers and adds each such chunk into the thread's own fp64 slots
        // in shared memory (a sum over many samples lost digits in fp32 where the terms cancel;
        // fp64 registers cost a resident block); an fp64 plan sums in registers.
        const bool dacc = R.wsh && !f64;
        if (R.wsh) {
            for (int pi = 0; pi < P->P; ++pi) S(fmt("%s dwa_%d = 0;", T.c_str(), pi));
            if (dacc) {
                S("double* const sacc = reinterpret_cast<double*>(smem + EG_DACC) + u;");
                S("int nacc = 0;");
                for (int g = 0; g < NG; ++g) {
                    std::string st;
                    for (int pi : P->groups[g]) st += fmt(" sacc[%d * UVU_UP] = 0.0;", pi);
                    S(fmt("%sif (g == %d) {%s }", g ? "else " : "", g, st.c_str()));
                }
            }
        }
        auto flush = [&](const char* cond) {
            S(std::string("if (") + cond + ") {");
            for (int g = 0; g < NG; ++g) {
                std::string st;
                for (int pi : P->groups[g]) st += fmt(" sacc[%d * UVU_UP] += (double)dwa_%d; dwa_%d = 0;", pi, pi, pi);
                S(fmt("  %sif (g == %d) {%s }", g ? "else " : "", g, st.c_str()));
            }
            S("}");
        };
        S("for (long long r = blockIdx.x; r < N; r += gridDim.x) {");
        S.ind++;
        S("const int e0 = " + off_at(R, "r") + ", e1 = " + off_at(R, "r + 1") + ";");
        for (int g = 0; g < NG; ++g) {
            std::string dwa;
            if (R.wsh)
                for (int pi : P->groups[g]) dwa += fmt(", dwa_%d", pi);
            S(fmt("%sif (g == %d) edge_rcv%d(r, e0, e1, u, uvalid, lane, warp, tid, c, kg, dead, buf, smem, sbase, src, x, Y, %sgout, dY, dw, dx, dxe, g, w%s);",
                  g ? "else " : "", g, g, R.dual ? "ax, aY, hm, " : "", dwa.c_str()));
        }
        if (dacc) flush("++nacc == 16 && (nacc = 0, true)");
        S.ind--;
        S("}");
        if (obulk) S("if (tid == 0) bulk_wait_all();  // the last stages' outputs are written");
        obulk = false;
        if (dacc) flush("true");
        if (R.wsh) {  // the block's partial dw [P][U] in fp64 (row blockIdx.x of the caller's workspace)
            S("if (dw && uvalid) {");
            S("  double* __restrict__ pr = reinterpret_cast<double*>(dw) + (size_t)blockIdx.x * (UVU_P * UVU_U) + u;");
            for (int g = 0; g < NG; ++g) {
                std::string st;
                for (int pi : P->groups[g]) st += dacc ? fmt(" pr[%d * UVU_U] = sacc[%d * UVU_UP];", pi, pi)
                                                       : fmt(" pr[%d * UVU_U] = dwa_%d;", pi, pi);
                S(fmt("  %sif (g == %d) {%s }", g ? "else " : "", g, st.c_str()));
            }
            S("}");
        }
        S.ind--;
        S("}");
        dw_accum = false;
    }

    // Per-edge dx contribution of this thread's channel, for the deterministic (staged) dx:
    // written straight to dxe[e][u][:] with one register group, otherwise into the stage's
    // shared-memory partials [buf][g][j][u][:] that the consumers sum over groups after the
    // stage barrier (fixed order).
    void emit_dx_edge_store(Src& S, const std::set<int>& xn, int NG) const {
        S("if (dxe) {");
        S.ind++;
        if (NG == 1) {
            if (obulk)  // where this thread read its x row, then out with the stage
                S(fmt("%s* dxer = reinterpret_cast<%s*>(const_cast<unsigned char*>(stg) + EG_XOFF) + (j * UVU_U + u) * UVU_DX;",
                      T.c_str(), T.c_str()));
            else
                S(T + "* __restrict__ dxer = dxe + ((size_t)e * UVU_U + u) * UVU_DX;");
            if (!f64 && P->Dx % 4 == 0) {
                for (int c = 0; c < P->Dx / 4; ++c) {
                    std::string v[4];
                    for (int i = 0; i < 4; ++i) v[i] = xn.count(4 * c + i) ? fmt("dxp_%d", 4 * c + i) : "0.0f";
                    S(fmt("reinterpret_cast<float4*>(dxer)[%d] = make_float4(%s, %s, %s, %s);", c, v[0].c_str(), v[1].c_str(),
                          v[2].c_str(), v[3].c_str()));
                }
            } else {
                for (int k = 0; k < P->Dx; ++k) S(fmt("dxer[%d] = %s;", k, xn.count(k) ? fmt("dxp_%d", k).c_str() : "0"));
            }
        } else {
            S(fmt("%s* xp = reinterpret_cast<%s*>(const_cast<unsigned char*>(smem) + EG_XPART) + ((size_t)((buf * UVU_G + g) * EG_CH + j) * UVU_UP + u) * UVU_DX;",
                  T.c_str(), T.c_str()));
            for (int k = 0; k < P->Dx; ++k) S(fmt("xp[%d] = %s;", k, xn.count(k) ? fmt("dxp_%d", k).c_str() : "0"));
        }
        S.ind--;
        S("}");
    }

    void emit_dx_atomics(Src& S, const std::set<int>& xn) const {
        if (!f64 && P->Dx % 4 == 0) {
            std::set<int> chunks;
            for (int k : xn) chunks.insert(k / 4);
            for (int c : chunks) {
                std::string v[4];
                for (int i = 0; i < 4; ++i) v[i] = xn.count(4 * c + i) ? fmt("dxp_%d", 4 * c + i) : "0.0f";
                S(fmt("red_add_v4(dxr + %d, %s, %s, %s, %s);", 4 * c, v[0].c_str(), v[1].c_str(), v[2].c_str(), v[3].c_str()));
            }
        } else {
            for (int k : xn) S(fmt("atomicAdd(dxr + %d, dxp_%d);", k, k));
        }
    }

    // Sender-stationary sum of the per-edge dx partials over the transposed CSR: one thread per
    // (sender, channel) adds its edges' rows in ascending edge-id order and writes dx once.
    // UVU_REDUCE_GROUP=n (a tuning switch, 1..16): edges per group of the dx reduction
    // UVU_REDUCE_MINB=n (a tuning switch): resident 256-thread blocks per SM the dx reduction's
    // register budget is sized for
    static int reduce_minb() {
        const char* e = std::getenv("UVU_REDUCE_MINB");
        return e ? std::max(1, std::min(8, std::atoi(e))) : 4;
    }
    static int reduce_group() {
        const char* e = std::getenv("UVU_REDUCE_GROUP");
        const int g = e ? std::atoi(e) : 8;
        return std::max(1, std::min(16, g));
    }
    // dx[s] = sum over the out-edges e of s, in ascending edge id, of the per-edge partials
    // dxe[e] (each a row of U x D_x values).  When a row is a whole number of 16-byte vectors
    // the row is summed as flat vectors, one thread per (sender, vector) (D_x = 9 rows: one
    // 16-byte load per edge instead of nine scalar ones); otherwise one thread per (sender,
    // channel) sums its D_x values.  Either way every output value is the same ordered sum.
    void emit_dx_reduce(Src& S) const {
        const int V = f64 ? 2 : 4;
        const bool flat = (P->U * P->Dx) % V == 0;
        const int per = flat ? P->U * P->Dx / V : P->U_pad;
        P->reduce_per_sender = per;
        const std::string TV = f64 ? "double2" : "float4";
        S(fmt("extern \"C\" __global__ void __launch_bounds__(256, %d) uvu_bwd_dx_reduce(long long N, const int* __restrict__ soff,",
              reduce_minb()));
        S(fmt("    const int* __restrict__ seid, const %s* __restrict__ dxe, %s* __restrict__ dx) {", T.c_str(), T.c_str()));
        S.ind++;
        S("const long long t = (long long)blockIdx.x * 256 + threadIdx.x;");
        S(fmt("const long long sn = t / %d;", per));
        S(fmt("const int c = (int)(t - sn * %d);", per));
        S(flat ? "if (sn >= N) return;" : "if (sn >= N || c >= UVU_U) return;");
        S("const int k0 = __ldg(soff + sn), k1 = __ldg(soff + sn + 1);");
        const int nacc = flat ? V : P->Dx;
        for (int k = 0; k < nacc; ++k) S(fmt("%s a_%d = 0;", T.c_str(), k));
        const bool vec = !flat && !f64 && P->Dx % 4 == 0;
        auto add_row = [&](const std::string& e) {
            if (flat) {
                S(fmt("{ const %s v = __ldg(reinterpret_cast<const %s*>(dxe + (size_t)(%s) * (UVU_U * UVU_DX)) + c);", TV.c_str(),
                      TV.c_str(), e.c_str()));
                if (f64) S("  a_0 += v.x; a_1 += v.y; }");
                else S("  a_0 += v.x; a_1 += v.y; a_2 += v.z; a_3 += v.w; }");
                return;
            }
            S(fmt("{ const %s* __restrict__ row = dxe + ((size_t)(%s) * UVU_U + c) * UVU_DX;", T.c_str(), e.c_str()));
            if (vec) {
                for (int q = 0; q < P->Dx / 4; ++q) {
                    S(fmt("  const float4 v%d = __ldg(reinterpret_cast<const float4*>(row) + %d);", q, q));
                    S(fmt("  a_%d += v%d.x; a_%d += v%d.y; a_%d += v%d.z; a_%d += v%d.w;", 4 * q, q, 4 * q + 1, q, 4 * q + 2, q,
                          4 * q + 3, q));
                }
            } else {
                for (int k = 0; k < P->Dx; ++k) S(fmt("  a_%d += __ldg(row + %d);", k, k));
            }
            S("}");
        };
        // groups of kG edges, the next group's edge ids loaded while the current group's rows
        // are read (one dependent round trip per group instead of two); the rows are added in
        // ascending edge order, so the sum is the same for any grouping
        const int kG = reduce_group();
        S("int k = k0;");
        {
            std::string ld;
            for (int i = 0; i < kG; ++i) ld += fmt("%sn%d = (k + %d < k1) ? __ldg(seid + k + %d) : 0", i ? ", " : "int ", i, i, i);
            S(ld + ";");
        }
        S("#pragma unroll 1");
        S(fmt("for (; k + %d <= k1; k += %d) {", kG, kG));
        S.ind++;
        {
            std::string cur;
            for (int i = 0; i < kG; ++i) cur += fmt("%se%d = n%d", i ? ", " : "const int ", i, i);
            S(cur + ";");
            for (int i = 0; i < kG; ++i) S(fmt("n%d = (k + %d < k1) ? __ldg(seid + k + %d) : 0;", i, kG + i, kG + i));
        }
        for (int i = 0; i < kG; ++i) add_row(fmt("e%d", i));
        S.ind--;
        S("}");
        S("for (; k < k1; ++k) {");
        S.ind++;
        S("const int e0 = __ldg(seid + k);");
        add_row("e0");
        S.ind--;
        S("}");
        if (flat) {
            if (f64) S("reinterpret_cast<double2*>(dx + (size_t)sn * (UVU_U * UVU_DX))[c] = make_double2(a_0, a_1);");
            else S("reinterpret_cast<float4*>(dx + (size_t)sn * (UVU_U * UVU_DX))[c] = make_float4(a_0, a_1, a_2, a_3);");
        } else {
            S(T + "* __restrict__ dxr = dx + ((size_t)sn * UVU_U + c) * UVU_DX;");
            for (int k = 0; k < P->Dx; ++k) S(fmt("dxr[%d] = a_%d;", k, k));
        }
        S.ind--;
        S("}");
    }

    // ------------------------------------------------------------------ sender-stationary dx
    struct SendPipe {
        int ut = 32, ntile = 1, ch = 1, nst = 2;
        bool ybulk = false;
        size_t wt = 0, gt = 0, w_off = 0, g_off = 0, y_off = 0, stage = 0, bar_off = 0, total = 0, tx = 0;
    };

    SendPipe send_pipe() const {
        SendPipe D;
        D.ut = std::min(P->U_pad, 128);
        D.ntile = P->U_pad / D.ut;
        D.ybulk = ybytes() % 16 == 0;
        D.wt = size_t(P->P) * D.ut * P->elem();
        D.gt = size_t(D.ut) * P->Do * P->elem();
        const size_t pe = D.wt + D.gt + (D.ybulk ? ybytes() : 0);
        D.ch = int(std::max<size_t>(1, std::min<size_t>(8, 32768 / pe)));
        D.w_off = 0;
        D.g_off = a16(D.ch * D.wt);
        D.y_off = D.g_off + a16(D.ch * D.gt);
        D.stage = D.y_off + (D.ybulk ? a16(D.ch * ybytes()) : 0);
        D.nst = 2;
        D.bar_off = D.nst * D.stage;
        D.total = D.bar_off + 16 * D.nst;
        D.tx = pe;
        return D;
    }

    // Requirements of the tiled copies: channel tiles start and end on 16-byte boundaries.
    bool send_pipe_ok(const SendPipe& D) const {
        return P->U % D.ut == 0 && (size_t(D.ut) * P->elem()) % 16 == 0 && D.gt % 16 == 0 &&
               (size_t(P->U) * P->Do * P->elem()) % 16 == 0;
    }

    void emit_dx_v2(Src& S, const SendPipe& D) const {
        std::vector<int> all;
        for (int p = 0; p < P->P; ++p) all.push_back(p);
        const std::set<int> xn = x_needed(all), yn = y_needed(all);
        S(fmt("#define DX_UT %d", D.ut));
        S(fmt("#define DX_NT %d", D.ntile));
        S(fmt("#define DX_CH %d", D.ch));
        S(fmt("#define DX_NST %d", D.nst));
        S(fmt("#define DX_STAGE %zu", D.stage));
        S(fmt("#define DX_GOFF %zu", D.g_off));
        S(fmt("#define DX_YOFF %zu", D.y_off));
        S(fmt("#define DX_BAR %zu", D.bar_off));
        S(fmt("#define DX_TX %zu", D.tx));
        S(fmt("#define DX_NCW %d", D.ut / 32));
        const int mb = std::min(minb(D.total), P->minb[2]);
        P->minb_eff[2] = mb;
        S(fmt("#define DX_MINB %d", mb));
        // producer
        S(fmt("__device__ __noinline__ void dx_producer(long long N, const int* __restrict__ soff, const int* __restrict__ seid,"));
        S(fmt("    const int* __restrict__ srecv, const %s* __restrict__ Y, const %s* __restrict__ w, const %s* __restrict__ gout,",
              T.c_str(), T.c_str(), T.c_str()));
        S("    unsigned sbase) {");
        S.ind++;
        S("unsigned c = 0;");
        S("bool dead = false;");
        // The edge ids and receivers of the next chunk are loaded before the current chunk's
        // copies are issued (the copies are asm statements with a memory clobber).
        S("for (long long it = blockIdx.x; it < N * DX_NT && !dead; it += gridDim.x) {");
        S.ind++;
        S("const long long sn = it / DX_NT;");
        S("const int u0 = (int)(it - sn * DX_NT) * DX_UT;");
        S("const int k0 = __ldg(soff + sn), k1 = __ldg(soff + sn + 1);");
        for (int j = 0; j < D.ch; ++j)
            S(fmt("int ev%d = 0, rv%d = 0; if (k0 + %d < k1) { ev%d = __ldg(seid + k0 + %d); rv%d = __ldg(srecv + k0 + %d); }", j, j,
                  j, j, j, j, j));
        S("for (int kb = k0; kb < k1; kb += DX_CH, ++c) {");
        S.ind++;
        S("const int kn = kb + DX_CH;");
        for (int j = 0; j < D.ch; ++j)
            S(fmt("int evn%d = 0, rvn%d = 0; if (kn + %d < k1) { evn%d = __ldg(seid + kn + %d); rvn%d = __ldg(srecv + kn + %d); }", j,
                  j, j, j, j, j, j));
        S("const unsigned st = c % DX_NST;");
        S("if (c >= DX_NST && !mbar_wait(sbase + DX_BAR + 8u * (DX_NST + st), ((c / DX_NST) - 1u) & 1u)) { dead = true; break; }");
        S("const int ne = min(DX_CH, k1 - kb);");
        S("const unsigned full = sbase + DX_BAR + 8u * st;");
        S("const unsigned stg = sbase + st * DX_STAGE;");
        S("mbar_expect_tx(full, (unsigned)ne * DX_TX);");
        for (int j = 0; j < D.ch; ++j) {
            S(fmt("if (%d < ne) {", j));
            S.ind++;
            S(fmt("const int e = ev%d, r = rv%d;", j, j));
            if (D.ut == P->U) {
                S(fmt("bulk_g2s(stg + %zuu, w + (size_t)e * (UVU_P * UVU_U), %zuu, full);", size_t(j) * D.wt, D.wt));
            } else {
                S("#pragma unroll 1");
                S(fmt("for (int p = 0; p < UVU_P; ++p) bulk_g2s(stg + %zuu + (unsigned)p * %zuu, w + ((size_t)e * UVU_P + p) * UVU_U + u0, %zuu, full);",
                      size_t(j) * D.wt, size_t(D.ut) * P->elem(), size_t(D.ut) * P->elem()));
            }
            S(fmt("bulk_g2s(stg + DX_GOFF + %zuu, gout + ((size_t)r * UVU_U + u0) * UVU_DO, %zuu, full);", size_t(j) * D.gt, D.gt));
            if (D.ybulk) S(fmt("bulk_g2s(stg + DX_YOFF + %zuu, Y + (size_t)e * UVU_DY, %zuu, full);", size_t(j) * ybytes(), ybytes()));
            S.ind--;
            S("}");
        }
        for (int j = 0; j < D.ch; ++j) S(fmt("ev%d = evn%d; rv%d = rvn%d;", j, j, j, j));
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S("if (dead) {");
        S("  const unsigned n = c < DX_NST ? c : DX_NST;");
        S("  for (unsigned k = c - n; k < c; ++k) mbar_wait(sbase + DX_BAR + 8u * (k % DX_NST), (k / DX_NST) & 1u);");
        S("}");
        S.ind--;
        S("}");
        // kernel
        S(fmt("extern \"C\" __global__ void __launch_bounds__(DX_UT + 32, DX_MINB) uvu_bwd_dx(long long N, const int* __restrict__ soff,"));
        S(fmt("    const int* __restrict__ seid, const int* __restrict__ srecv, const %s* __restrict__ Y,", T.c_str()));
        S(fmt("    const %s* __restrict__ w, const %s* __restrict__ gout, %s* __restrict__ dx) {", T.c_str(), T.c_str(), T.c_str()));
        S.ind++;
        S("extern __shared__ __align__(128) unsigned char smem[];");
        S("const unsigned sbase = smem_addr(smem);");
        S("const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;");
        S("if (tid == 0) {");
        S("  for (int i = 0; i < DX_NST; ++i) { mbar_init(sbase + DX_BAR + 8u * i, 1u); mbar_init(sbase + DX_BAR + 8u * (DX_NST + i), " + std::string(empty_count("DX_NCW", "DX_UT")) + "); }");
        S("  asm volatile(\"fence.mbarrier_init.release.cluster;\" ::: \"memory\");");
        S("}");
        S("__syncthreads();");
        S("if (warp == DX_NCW) {");
        S("  if (lane == 0) dx_producer(N, soff, seid, srecv, Y, w, gout, sbase);");
        S("  return;");
        S("}");
        S("const int ul = tid;");
        S("unsigned c = 0;");
        S("bool dead = false;");
        S("for (long long it = blockIdx.x; it < N * DX_NT; it += gridDim.x) {");
        S.ind++;
        S("const long long sn = it / DX_NT;");
        S("const int u = (int)(it - sn * DX_NT) * DX_UT + ul;");
        S("const bool uvalid = u < UVU_U;");
        S("const int k0 = __ldg(soff + sn), k1 = __ldg(soff + sn + 1);");
        for (int k : xn) S(fmt("%s dxp_%d = 0;", T.c_str(), k));
        S("for (int kb = k0; kb < k1; kb += DX_CH, ++c) {");
        S.ind++;
        S("const unsigned st = c % DX_NST;");
        S("if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(sbase + DX_BAR + 8u * st, (c / DX_NST) & 1u));");
        S("if (dead) continue;");
        S("const int ne = min(DX_CH, k1 - kb);");
        S("const unsigned char* stg = smem + st * DX_STAGE;");
        S("if (uvalid) {");
        S.ind++;
        S("#pragma unroll");
        S("for (int j = 0; j < DX_CH; ++j) {");
        S.ind++;
        S("if (j < ne) {");
        S.ind++;
        if (D.ybulk)
            emit_row_loads(S, "yv", fmt("reinterpret_cast<const %s*>(stg + DX_YOFF) + j * UVU_DY", T.c_str()), P->Dy, yn, false);
        else {
            S("const int e = __ldg(seid + kb + j);");
            emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
        }
        S(fmt("const %s* swr = reinterpret_cast<const %s*>(stg) + j * (UVU_P * DX_UT) + ul;", T.c_str(), T.c_str()));
        for (int pi : all) S(fmt("const %s wv_%d = swr[%d * DX_UT];", T.c_str(), pi, pi));
        S(fmt("const %s* sgr = reinterpret_cast<const %s*>(stg + DX_GOFF) + (j * DX_UT + ul) * UVU_DO;", T.c_str(), T.c_str()));
        auto gval = [](int k) { return fmt("sgr[%d]", k); };
        emit_bwd_pairs(S, all, false, false, true, gval);
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        emit_release(S, "DX");
        S.ind--;
        S("}");
        S("if (uvalid) {");
        S.ind++;
        S(T + "* __restrict__ dxr = dx + ((size_t)sn * UVU_U + u) * UVU_DX;");
        for (int k = 0; k < P->Dx; ++k) S(fmt("dxr[%d] = %s;", k, xn.count(k) ? fmt("dxp_%d", k).c_str() : "0"));
        S.ind--;
        S("}");
        S.ind--;
        S("}");
        S.ind--;
        S("}");
    }

    // ------------------------------------------------------------------ fused radial forward
    // Forward with the radial weights formed in registers: w[e,p,u] = sum_k h[e,k] W_last[k,p,u]
    // for the NE edges a thread takes together, then the receiver-stationary contraction of each
    // edge ("Receiver-streaming convolutions for channel-wise UVU tensor products", replies: the
    // radial network fused into the convolution instead of its weights read from memory).
    // One warp = one receiver x 32 channels x one register group; a block's warps share a slice of
    // 32 channels, whose last-layer weights [H][P][32] sit in shared memory when they fit (else
    // they are read through the read-only cache).  Forming NE edges' weights together reuses each
    // last-layer weight NE times from a register.
    mutable int radial_h_ = 0;  // hidden width of the radial module being emitted
    int H_bytes_lines() const { return int((size_t(radial_h_) * P->elem() + 127) / 128); }
    // packed: fp32 weights formed two paths at a time with the paired FMA (fma.rn.f32x2), the
    // last layer staged as (even, odd) path pairs per lane; each half rounds as a scalar FMA.
    // split: the block holds only this group's path pairs [q0, q0 + gp) of the last layer
    void emit_radial_group(Src& S, int g, const std::vector<int>& paths, int NE, bool packed, bool split = false) const {
        const std::set<int> xn = x_needed(paths), yn = y_needed(paths);
        std::vector<int> outs;
        for (int pi : paths)
            for (int m = 0; m < 2 * P->paths[pi].l3 + 1; ++m) outs.push_back(P->paths[pi].ooff + m);
        std::set<int> pairs;
        for (int pi : paths) pairs.insert(pi / 2);
        const bool f = !f64;
        S(fmt("__device__ __forceinline__ void rad_group%d(int e0, int e1, const int* __restrict__ src, const %s* __restrict__ x,", g, T.c_str()));
        S(fmt("    const %s* __restrict__ Y, const %s* __restrict__ h, const %s* __restrict__ wlb, int u, %s* __restrict__ orow) {",
              T.c_str(), T.c_str(), T.c_str(), T.c_str()));
        S.ind++;
        for (int k : outs) S(fmt("%s acc_%d = 0;", T.c_str(), k));
        S("#pragma unroll 1");
        S("for (int eb = e0; eb < e1; eb += RD_NE) {");
        S.ind++;
        S("const int ne = min(RD_NE, e1 - eb);");
        // the batch's sender ids, and its x and Y rows asked into L1 before the weights are
        // formed (UVU_RAD_PREFETCH=0, a tuning switch, leaves them to the loads after)
        // (UVU_RAD_PREFETCH=2 also asks for the next batch's h rows)
        const int pfm = std::getenv("UVU_RAD_PREFETCH") ? std::atoi(std::getenv("UVU_RAD_PREFETCH")) : 1;
        const bool pf = pfm != 0;
        for (int j = 0; j < NE; ++j) S(fmt("const int s%d = __ldg(src + eb + min(%d, ne - 1));", j, j));
        if (pf)
            for (int j = 0; j < NE; ++j) {
                S(fmt("prefetch_l1(x + ((size_t)s%d * UVU_U + u) * UVU_DX);", j));
                S(fmt("prefetch_l1(Y + (size_t)(eb + min(%d, ne - 1)) * UVU_DY);", j));
            }
        if (pfm == 2) {
            S("if (eb + RD_NE < e1) {");
            for (int j = 0; j < NE; ++j)
                for (int b = 0; b < H_bytes_lines(); ++b)
                    S(fmt("  prefetch_l1(reinterpret_cast<const char*>(h + (size_t)min(eb + RD_NE + %d, e1 - 1) * RD_H) + %d);", j, b * 128));
            S("}");
        }
        for (int j = 0; j < NE; ++j) {
            S(fmt("const %s* __restrict__ hr%d = h + (size_t)(eb + min(%d, ne - 1)) * RD_H;", T.c_str(), j, j));
            if (packed)
                for (int q : pairs) S(fmt("unsigned long long w%d_q%d = 0;", j, q));
            else
                for (int pi : paths) S(fmt("%s w%d_%d = 0;", T.c_str(), j, pi));
        }
        S("#pragma unroll 2");
        S("for (int k = 0; k < RD_H; k += 4) {");
        S.ind++;
        static const char* comp[4] = {"x", "y", "z", "w"};
        for (int j = 0; j < NE; ++j) {
            if (f) {
                S(fmt("const float4 hq%d = __ldg(reinterpret_cast<const float4*>(hr%d + k));", j, j));
            } else {
                S(fmt("const double2 hqa%d = __ldg(reinterpret_cast<const double2*>(hr%d + k));", j, j));
                S(fmt("const double2 hqb%d = __ldg(reinterpret_cast<const double2*>(hr%d + k) + 1);", j, j));
            }
        }
        if (packed) {
            const int q0 = split ? *pairs.begin() : 0;
            const int gp = split ? int(pairs.size()) : (P->P + 1) / 2;
            S(fmt("const unsigned long long* __restrict__ wk = reinterpret_cast<const unsigned long long*>(wlb) + (size_t)k * (%s * 32);",
                  split ? fmt("%d", gp).c_str() : "RD_P2"));
            for (int kk = 0; kk < 4; ++kk) {
                for (int j = 0; j < NE; ++j) S(fmt("const unsigned long long hp%d_%d = f2pack(hq%d.%s, hq%d.%s);", j, kk, j, comp[kk], j, comp[kk]));
                for (int q : pairs) {
                    S(fmt("{ const unsigned long long wl = wk[%d * 32];", kk * gp + (q - q0)));
                    for (int j = 0; j < NE; ++j) S(fmt("  w%d_q%d = ffma2(hp%d_%d, wl, w%d_q%d);", j, q, j, kk, j, q));
                    S("}");
                }
            }
        } else {
            S(fmt("const %s* __restrict__ wk = wlb + (size_t)k * (UVU_P * RD_WSTR);", T.c_str()));
            for (int kk = 0; kk < 4; ++kk) {
                for (int pi : paths) {
                    S(fmt("{ const %s wl = wk[%d * RD_WSTR];", T.c_str(), kk * P->P + pi));
                    for (int j = 0; j < NE; ++j) {
                        const std::string hv = f ? fmt("hq%d.%s", j, comp[kk]) : fmt("hq%c%d.%s", kk < 2 ? 'a' : 'b', j, comp[kk % 2]);
                        S(fmt("  w%d_%d = fma(%s, wl, w%d_%d);", j, pi, hv.c_str(), j, pi));
                    }
                    S("}");
                }
            }
        }
        S.ind--;
        S("}");
        for (int j = 0; j < NE; ++j) {
            S(fmt("if (%d < ne) {", j));
            S.ind++;
            S(fmt("const int e = eb + %d;", j));
            emit_row_loads(S, "xv", fmt("x + ((size_t)s%d * UVU_U + u) * UVU_DX", j), P->Dx, xn);
            emit_row_loads(S, "yv", "Y + (size_t)e * UVU_DY", P->Dy, yn);
            if (packed) {
                for (int q : pairs) S(fmt("float wq%d_a, wq%d_b; f2unpack(w%d_q%d, wq%d_a, wq%d_b);", q, q, j, q, q, q));
                for (int pi : paths) S(fmt("const float wv_%d = wq%d_%c;", pi, pi / 2, pi % 2 ? 'b' : 'a'));
            } else {
                for (int pi : paths) S(fmt("const %s wv_%d = w%d_%d;", T.c_str(), pi, j, pi));
            }
            emit_fwd_edge(S, paths);
            S.ind--;
            S("}");
        }
        S.ind--;
        S("}");
        for (int k : outs) S(fmt("orow[%d] = acc_%d;", k, k));
        S.ind--;
        S("}");
    }

    // split: one block per (channel slice, register group), holding that group's pairs only
    void emit_fwd_radial(Src& S, const std::vector<std::vector<int>>& rg, int NE, bool packed, bool split = false) const {
        const int NG = int(rg.size());
        S("__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile(\"prefetch.global.L1 [%0];\" :: \"l\"(p)); }");
        if (packed) {
            S("__device__ __forceinline__ unsigned long long f2pack(float a, float b) {");
            S("  unsigned long long r; asm(\"mov.b64 %0, {%1, %2};\" : \"=l\"(r) : \"f\"(a), \"f\"(b)); return r; }");
            S("__device__ __forceinline__ void f2unpack(unsigned long long v, float& a, float& b) {");
            S("  asm(\"mov.b64 {%0, %1}, %2;\" : \"=f\"(a), \"=f\"(b) : \"l\"(v)); }");
            S("// two fp32 FMAs in one instruction, each rounded as fmaf");
            S("__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {");
            S("  unsigned long long d; asm(\"fma.rn.f32x2 %0, %1, %2, %3;\" : \"=l\"(d) : \"l\"(a), \"l\"(b), \"l\"(c)); return d; }");
        }
        for (int g = 0; g < NG; ++g) emit_radial_group(S, g, rg[g], NE, packed, split);
        if (split) {
            emit_fwd_radial_split(S, rg);
            return;
        }
        S(fmt("extern \"C\" __global__ void __launch_bounds__(RD_TPB, RD_MINB) uvu_fwd_radial(long long N, const int* __restrict__ off,"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y, const %s* __restrict__ h,",
              T.c_str(), T.c_str(), T.c_str()));
        S(fmt("    const %s* __restrict__ wlast, %s* __restrict__ out) {", T.c_str(), T.c_str()));
        S.ind++;
        S("const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;");
        S("const int sl = blockIdx.x % RD_NSL;");
        S("const long long rb = blockIdx.x / RD_NSL, nbs = gridDim.x / RD_NSL;");
        S("const int u = sl * 32 + lane;");
        S("#if RD_WSM");
        S("extern __shared__ __align__(16) unsigned char smem[];");
        S(fmt("%s* const wls = reinterpret_cast<%s*>(smem);", T.c_str(), T.c_str()));
        if (packed) {  // [k][path pair][lane][2]; the odd path past the last is zero
            S("for (int i = threadIdx.x; i < RD_H * RD_P2 * 64; i += RD_TPB) {");
            S("  const int l = (i >> 1) & 31, uu = sl * 32 + l, kq = i >> 6, k = kq / RD_P2, p = 2 * (kq - k * RD_P2) + (i & 1);");
            S("  wls[i] = (uu < UVU_U && p < UVU_P) ? __ldg(wlast + ((size_t)k * UVU_P + p) * UVU_U + uu) : 0;");
            S("}");
        } else {  // [k][path][lane]
            S("for (int i = threadIdx.x; i < RD_H * UVU_P * 32; i += RD_TPB) {");
            S("  const int l = i & 31, uu = sl * 32 + l;");
            S("  wls[i] = uu < UVU_U ? __ldg(wlast + (size_t)(i >> 5) * UVU_U + uu) : 0;");
            S("}");
        }
        S("__syncthreads();");
        S(fmt("const %s* const wlb = wls + %s;", T.c_str(), packed ? "2 * lane" : "lane"));
        S("#else");
        S(fmt("const %s* const wlb = wlast + u;", T.c_str()));
        S("#endif");
        S("if (u >= UVU_U || rb >= nbs) return;");
        S("const int g = warp % RD_NG;");
        S("for (long long r = rb * RD_RPB + warp / RD_NG; r < N; r += nbs * RD_RPB) {");
        S.ind++;
        S("const int e0 = __ldg(off + r), e1 = __ldg(off + r + 1);");
        S(fmt("%s* const orow = out + ((size_t)r * UVU_U + u) * UVU_DO;", T.c_str()));
        for (int g = 0; g < NG; ++g)
            S(fmt("%sif (g == %d) rad_group%d(e0, e1, src, x, Y, h, wlb, u, orow);", g ? "else " : "", g, g));
        S.ind--;
        S("}");
        S.ind--;
        S("}");
    }
    void emit_fwd_radial_split(Src& S, const std::vector<std::vector<int>>& rg) const {
        const int NG = int(rg.size());
        S(fmt("extern \"C\" __global__ void __launch_bounds__(RD_TPB, RD_MINB) uvu_fwd_radial(long long N, const int* __restrict__ off,"));
        S("    const int* __restrict__ src, const float* __restrict__ x, const float* __restrict__ Y, const float* __restrict__ h,");
        S("    const float* __restrict__ wlast, float* __restrict__ out) {");
        S.ind++;
        S("const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;");
        S("const int sl = blockIdx.x % RD_NSL, g = (blockIdx.x / RD_NSL) % RD_NG;");
        S("const long long rb = blockIdx.x / (RD_NSL * RD_NG), nbs = gridDim.x / (RD_NSL * RD_NG);");
        S("const int u = sl * 32 + lane;");
        S("extern __shared__ __align__(16) unsigned char smem[];");
        S("float* const wls = reinterpret_cast<float*>(smem);");
        std::string q0s = "{", gps = "{";
        for (int g = 0; g < NG; ++g) {
            std::set<int> pr;
            for (int pi : rg[g]) pr.insert(pi / 2);
            q0s += fmt("%s%d", g ? ", " : "", *pr.begin());
            gps += fmt("%s%d", g ? ", " : "", int(pr.size()));
        }
        S(fmt("const int q0s[RD_NG] = %s}, gps[RD_NG] = %s};", q0s.c_str(), gps.c_str()));
        S("const int q0 = q0s[g], gp = gps[g];");
        S("// [k][pair of this group][lane][2]; a path past the last is zero");
        S("for (int i = threadIdx.x; i < RD_H * gp * 64; i += RD_TPB) {");
        S("  const int l = (i >> 1) & 31, uu = sl * 32 + l, kq = i >> 6, k = kq / gp, p = 2 * (q0 + kq - k * gp) + (i & 1);");
        S("  wls[i] = (uu < UVU_U && p < UVU_P) ? __ldg(wlast + ((size_t)k * UVU_P + p) * UVU_U + uu) : 0.f;");
        S("}");
        S("__syncthreads();");
        S("const float* const wlb = wls + 2 * lane;");
        S("if (u >= UVU_U || rb >= nbs) return;");
        S("for (long long r = rb * RD_RPB + warp; r < N; r += nbs * RD_RPB) {");
        S.ind++;
        S("const int e0 = __ldg(off + r), e1 = __ldg(off + r + 1);");
        S("float* const orow = out + ((size_t)r * UVU_U + u) * UVU_DO;");
        for (int g = 0; g < NG; ++g)
            S(fmt("%sif (g == %d) rad_group%d(e0, e1, src, x, Y, h, wlb, u, orow);", g ? "else " : "", g, g));
        S.ind--;
        S("}");
        S.ind--;
        S("}");
    }
};

}  // namespace

// Split the paths into `ng` contiguous register groups of about equal per-edge cost (CG
// non-zeros plus two operations per output component).
void balance_groups(Plan* plan, int ng) {
    std::vector<double> cost;
    double total = 0;
    for (const PathInfo& p : plan->paths) {
        cost.push_back(double(p.nz.size()) + 2.0 * (2 * p.l3 + 1));
        total += cost.back();
    }
    plan->groups.assign(1, {});
    double acc = 0;
    for (int p = 0; p < plan->P; ++p) {
        const int g = int(plan->groups.size()) - 1;
        if (!plan->groups.back().empty() && g + 1 < ng && acc + cost[p] / 2 > total * (g + 1) / ng)
            plan->groups.emplace_back();
        plan->groups.back().push_back(p);
        acc += cost[p];
    }
}

std::string emit_source(Plan* plan) {
    Gen G{plan, plan->dtype == UVU_F64, plan->dtype == UVU_F64 ? "double" : "float"};
    const int U = plan->U, NG = int(plan->groups.size());
    // Channel slots per owner: U rounded up to a whole number of warps (or, below 32, to a power
    // of two dividing 32) so that no warp mixes two owners; padding lanes hold no channel.
    int UP = 1;
    if (U >= 32) UP = (U + 31) / 32 * 32;
    else while (UP < U) UP *= 2;
    plan->U_pad = UP;
    const int owner_threads = UP * NG;
    const int rpb = std::max(1, 128 / owner_threads);
    const int segw = std::min(UP, 32);
    const int segs = NG * ((UP + 31) / 32);
    const int spb = std::max(1, 128 / UP);
    const int ch = 16;
    const int ncw = NG * UP / 32;

    // Pipelined (bulk-copy) kernels need whole warps per owner and 16-byte multiples for the
    // per-edge weight rows; otherwise the direct-load kernels are emitted.  For the pipelined
    // kernels the paths are re-split into register groups of balanced per-edge cost so that an
    // owner has at least 8 consumer warps (more warps to hide shared-memory and FMA latency).
    // UVU_FORCE_DIRECT=1 (a debugging switch) selects the direct-load kernels everywhere.
    const bool force_direct = std::getenv("UVU_FORCE_DIRECT") && std::atoi(std::getenv("UVU_FORCE_DIRECT")) != 0;
    bool pipe_recv = !force_direct && U >= 32 && G.wbytes() % 16 == 0 && ncw * 32 + 32 <= 1024;
    // UVU_PIPE_GROUPS=n (a tuning switch) re-splits the paths into n register groups of
    // balanced per-edge cost for the pipelined kernels; by default the register-budget groups
    // stand (more groups add a barrier-coupled imbalance between warps that measured slower).
    if (pipe_recv && std::getenv("UVU_PIPE_GROUPS") && !plan->rebalanced) {
        const int ng2 = std::max(1, std::min(std::min(plan->P, std::atoi(std::getenv("UVU_PIPE_GROUPS"))), std::max(1, 512 / UP)));
        if (ng2 != NG) {
            balance_groups(plan, ng2);
            plan->rebalanced = true;
            return emit_source(plan);  // once more, with the new grouping
        }
    }
    // UVU_PIPE_OSTAGE=0 (a tuning switch) writes the forward output straight from registers.
    const bool ostage = !(std::getenv("UVU_PIPE_OSTAGE") && std::atoi(std::getenv("UVU_PIPE_OSTAGE")) == 0);
    // UVU_PIPE_GSTAGE=0 (a tuning switch) reads the edge kernel's d_out rows straight from global memory.
    const bool gstage = !(std::getenv("UVU_PIPE_GSTAGE") && std::atoi(std::getenv("UVU_PIPE_GSTAGE")) == 0);
    Gen::RecvPipe RF = G.fwd_pipe(ncw, plan->minb[0], ostage), RE = G.recv_pipe(true, ncw, false, 0, gstage);
    // Edge kernel: with a wide d_out row (fp32, D_out > 64) the row is read from the staged block
    // at each use rather than held in registers, and each (x irrep, SH irrep) pair is emitted in
    // one pass (MACE-large: 255 -> 168 registers, two resident blocks instead of one, edge kernel
    // 2.64 -> 2.53 ms; wide: spills gone, 5.85 -> 5.66 ms; measured slower on MACE-medium, 0.82 ->
    // 0.89 ms, and on the fp64 workload).  UVU_PIPE_GSMEM=1/0 (a tuning switch) forces it on or off.
    {
        bool gsm = plan->Do > 64 && plan->dtype == UVU_F32;
        if (const char* e = std::getenv("UVU_PIPE_GSMEM")) gsm = std::atoi(e) != 0;
        RE.gsm = RE.gst && !RE.lastwarp && gsm;
    }
    Gen::SendPipe SD = G.send_pipe();
    const bool pipe_dx = !force_direct && U >= 32 && G.send_pipe_ok(SD);
    plan->pipelined_recv = pipe_recv;
    plan->pipelined_dx = pipe_dx;
    if (pipe_recv) {
        plan->g_fwd = {ncw * 32 + 32, 1, RF.total, true};
        plan->g_edge = {ncw * 32 + 32, 1, RE.total, true};
    } else {
        plan->g_fwd = {rpb * owner_threads, rpb, 0, false};
        plan->g_edge = {rpb * owner_threads, rpb, size_t(rpb) * segs * ch * plan->Dy * plan->elem(), false};
    }
    plan->edge_chunk = pipe_recv ? RE.ch : ch;
    const int fs_spb = std::max(1, 128 / owner_threads);
    plan->g_fwd_sender = {fs_spb * owner_threads, fs_spb, 0, false};
    if (pipe_dx)
        plan->g_dx = {SD.ut + 32, 1, SD.total, true, SD.ntile};
    else
        plan->g_dx = {spb * UP, spb, 0, false};

    Src S;
    S("// Generated by the UVU planner. Channel-wise CG tensor-product graph convolution.");
    S(fmt("// irreps_x=%s irreps_sh=%s lmax_out=%d dtype=%s", plan->irreps_x.c_str(),
          plan->irreps_sh.c_str(), plan->lmax_out, G.f64 ? "fp64" : "fp32"));
    for (int p = 0; p < plan->P; ++p) {
        const PathInfo& pi = plan->paths[p];
        S(fmt("// path %d: (%d,%d,%d) parity %+d xoff %d yoff %d ooff %d nnz %zu", p, pi.l1, pi.l2,
              pi.l3, pi.parity, pi.xoff, pi.yoff, pi.ooff, pi.nz.size()));
    }
    S(fmt("#define UVU_U %d", U));
    S(fmt("#define UVU_UP %d", UP));
    S(fmt("#define UVU_P %d", plan->P));
    S(fmt("#define UVU_DX %d", plan->Dx));
    S(fmt("#define UVU_DY %d", plan->Dy));
    S(fmt("#define UVU_DO %d", plan->Do));
    S(fmt("#define UVU_G %d", NG));
    S(fmt("#define UVU_RPB %d", rpb));
    S(fmt("#define UVU_TPB %d", rpb * owner_threads));
    S(fmt("#define UVU_SEGW %d", segw));
    S(fmt("#define UVU_SEGS %d", segs));
    S(fmt("#define UVU_CH %d", ch));
    S(fmt("#define UVU_SPB %d", spb));
    S(fmt("#define UVU_DX_TPB %d", spb * UP));
    S(fmt("#define UVU_NCW %d", ncw));
    S(fmt("#define UVU_NCT %d", ncw * 32));
    S(fmt("#define UVU_FS_SPB %d", fs_spb));
    S(fmt("#define UVU_FS_TPB %d", fs_spb * owner_threads));
    S("// Block-wide barrier usable from the per-group code paths: the non-aligned form may be");
    S("// reached from different call sites, as long as every thread of the block arrives the same");
    S("// number of times (each group runs the same uniform chunk loop).");
    S("__device__ __forceinline__ void block_sync() { asm volatile(\"barrier.sync 0;\" ::: \"memory\"); }");
    S("__device__ __forceinline__ void red_add_v4(float* a, float p, float q, float r, float s) {");
    S("  asm volatile(\"red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\" :: \"l\"(a), \"f\"(p), \"f\"(q), \"f\"(r), \"f\"(s) : \"memory\");");
    S("}");
    G.emit_pair_helpers(S);
    G.emit_pipe_helpers(S);
    if (pipe_recv) {
        G.emit_recv_pipe_defines(S, RF, "FW", plan->minb[0], plan->minb_eff[0]);
        G.emit_recv_pipe_defines(S, RE, "EG", plan->minb[1], plan->minb_eff[1]);
        G.emit_fwd_v2(S, RF);
        G.emit_edge_v2(S, RE);
    } else {
        for (int g = 0; g < NG; ++g) G.emit_fwd_group(S, g);
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_TPB) uvu_fwd(long long N, const int* __restrict__ off,"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y,", G.T.c_str(), G.T.c_str()));
        S(fmt("    const %s* __restrict__ w, %s* __restrict__ out) {", G.T.c_str(), G.T.c_str()));
        S("  const int u = threadIdx.x % UVU_UP;");
        S("  const int g = (threadIdx.x / UVU_UP) % UVU_G;");
        S("  const long long r = (long long)blockIdx.x * UVU_RPB + threadIdx.x / (UVU_UP * UVU_G);");
        S("  if (r >= N || u >= UVU_U) return;");
        S("  const int e0 = __ldg(off + r), e1 = __ldg(off + r + 1);");
        S("  " + G.T + "* orow = out + ((size_t)r * UVU_U + u) * UVU_DO;");
        for (int g = 0; g < NG; ++g)
            S(fmt("  %sif (g == %d) fwd_group%d(e0, e1, u, src, x, Y, w, orow);", g ? "else " : "", g, g));
        S("}");

        for (int g = 0; g < NG; ++g) G.emit_edge_group(S, g);
        S(fmt("extern \"C\" __global__ void __launch_bounds__(UVU_TPB) uvu_bwd_edge(long long N, const int* __restrict__ off,"));
        S(fmt("    const int* __restrict__ src, const %s* __restrict__ x, const %s* __restrict__ Y,", G.T.c_str(), G.T.c_str()));
        S(fmt("    const %s* __restrict__ w, const %s* __restrict__ gout, %s* __restrict__ dY, %s* __restrict__ dw,",
              G.T.c_str(), G.T.c_str(), G.T.c_str(), G.T.c_str()));
        S(fmt("    %s* __restrict__ dx, %s* __restrict__ dxe) {", G.T.c_str(), G.T.c_str()));
        S(fmt("  extern __shared__ __align__(16) unsigned char smem_raw[];"));
        S(fmt("  %s* sred = reinterpret_cast<%s*>(smem_raw);", G.T.c_str(), G.T.c_str()));
        S("  __shared__ int s_e0[UVU_RPB], s_e1[UVU_RPB], s_nch;");
        S("  const int u = threadIdx.x % UVU_UP;");
        S("  const int g = (threadIdx.x / UVU_UP) % UVU_G;");
        S("  const int rl = threadIdx.x / (UVU_UP * UVU_G);");
        S("  const long long r = (long long)blockIdx.x * UVU_RPB + rl;");
        S("  const bool rvalid = r < N;");
        S("  const bool valid = rvalid && u < UVU_U;");
        S("  if (threadIdx.x == 0) s_nch = 0;");
        S("  __syncthreads();");
        S("  if (threadIdx.x % (UVU_UP * UVU_G) == 0) {");
        S("    const int a = rvalid ? __ldg(off + r) : 0, b = rvalid ? __ldg(off + r + 1) : 0;");
        S("    s_e0[rl] = a; s_e1[rl] = b;");
        S("    atomicMax(&s_nch, (b - a + UVU_CH - 1) / UVU_CH);");
        S("  }");
        S("  __syncthreads();");
        S("  const int nchunks = s_nch;");
        S("  const int seg = g * ((UVU_UP + 31) / 32) + u / 32;");
        S("  const int lane_in_seg = u % UVU_SEGW;");
        for (int g = 0; g < NG; ++g)
            S(fmt("  %sif (g == %d) edge_group%d(rl, seg, lane_in_seg, valid, s_e0[rl], s_e1[rl], nchunks, r, u, src, x, Y, w, gout, dY, dw, dx, sred, s_e0, s_e1, dxe);",
                  g ? "else " : "", g, g));
        S("}");
    }
    if (pipe_dx)
        G.emit_dx_v2(S, SD);
    else
        G.emit_dx_kernel(S);
    G.emit_dx_reduce(S);
    G.emit_fwd_sender_kernel(S);
    plan->staged_ok = pipe_recv || NG == 1;
    return S.o.str();
}

}  // namespace uvu

namespace uvu {

// Source of the plan's second module: the double-backward (HVP) kernels, compiled on the first
// HVP call so that plans used only for the forward and the VJP do not pay for them.  They use
// the direct-load structure and the plan's register groups.
const char* const kAuxKernelNames[AUX_COUNT][2] = {
    {"uvu_hvp_fwd", "uvu_hvp_edge"}, {"uvu_tp_fwd", "uvu_tp_edge"}, {"uvu_tp_fwd_sh", "uvu_tp_edge_sh"},
    {"uvu_fwd_radial", nullptr}};

namespace {
// Source of the fused-radial-weight forward for hidden width A.radial_h.  Register groups: runs
// of consecutive paths whose accumulators plus the NE edges' weights fit one thread's budget
// (UVU_RAD_BUDGET, a tuning switch, overrides it).  Warps per block: a multiple of the group
// count near six (two blocks per SM: twelve warps of up to 168 registers), twelve when the
// last-layer slice leaves room for one block per SM only.  Measured on MACE-medium (hidden 64):
// three edges per thread with twelve warps per SM ran 1.89 ms, against 2.22 ms for two edges
// with sixteen warps (128 registers) and 1.96 ms for four edges with twelve warps; the
// shared-memory reads of the last layer (one per FMA / NE) bound the two-edge form.
std::string emit_radial_source(Plan* plan) {
    Gen G{plan, plan->dtype == UVU_F64, plan->dtype == UVU_F64 ? "double" : "float"};
    AuxBuild& A = plan->aux[AUX_RADIAL];
    const int NE = A.radial_ne, H = A.radial_h;
    int budget = G.f64 ? 64 : 128;
    if (const char* e = std::getenv("UVU_RAD_BUDGET")) budget = std::max(8, std::atoi(e));
    std::vector<std::vector<int>> rg(1);
    int width = 0;
    for (int p = 0; p < plan->P; ++p) {
        const int c = 2 * plan->paths[p].l3 + 1 + NE;
        if (!rg.back().empty() && width + c > budget) {
            rg.emplace_back();
            width = 0;
        }
        rg.back().push_back(p);
        width += c;
    }
    // fp32 plans pair the paths (UVU_RAD_PACK=0, a tuning switch, keeps one path per FMA)
    const int P2 = (plan->P + 1) / 2;
    const bool pack_ok = !G.f64 && !(std::getenv("UVU_RAD_PACK") && std::atoi(std::getenv("UVU_RAD_PACK")) == 0);
    const size_t wsm_packed = size_t(H) * P2 * 64 * plan->elem();
    const size_t wsm_plain = size_t(H) * plan->P * 32 * plan->elem();
    const bool packed = pack_ok && wsm_packed <= 200 * 1024 + 16 * 1024;
    // UVU_RAD_SPLIT=n (a tuning switch): the paths in n runs of whole pairs, one block per (channel
    // slice, run), each block holding its run's part of the last layer only
    const int split_n = (packed && std::getenv("UVU_RAD_SPLIT")) ? std::min(P2, std::atoi(std::getenv("UVU_RAD_SPLIT"))) : 0;
    if (split_n >= 2) {
        rg.assign(split_n, {});
        for (int p = 0; p < plan->P; ++p) rg[std::min(split_n - 1, ((p / 2) * 2 + 1) * split_n / (2 * P2))].push_back(p);
        size_t gpmax = 0;
        for (auto& v : rg) gpmax = std::max<size_t>(gpmax, (v.back() / 2) - (v.front() / 2) + 1);
        const size_t smem = size_t(H) * gpmax * 64 * plan->elem();
        const int fit = int(std::min<size_t>(8, (227 * 1024) / (smem + 1024)));
        int rw = 6;
        if (const char* e = std::getenv("UVU_RAD_RW")) rw = std::max(1, std::min(32, std::atoi(e)));
        const int minb = std::max(1, std::min({fit, A.minb[0], 2048 / (rw * 32)}));
        A.minb_eff[0] = minb;
        A.radial_wsm = true;
        A.radial_nsl = (plan->U + 31) / 32;
        A.radial_rpb = rw;
        A.radial_gblk = split_n;
        A.g[0] = {rw * 32, 1, smem, true};
        A.g[1] = {};
        Src S;
        S("// Generated by the UVU planner: forward with fused radial weights (last layer in registers),");
        S("// one block per (channel slice, run of path pairs).");
        S(fmt("// irreps_x=%s irreps_sh=%s lmax_out=%d dtype=fp32 hidden=%d", plan->irreps_x.c_str(), plan->irreps_sh.c_str(),
              plan->lmax_out, H));
        S(fmt("#define UVU_U %d", plan->U));
        S(fmt("#define UVU_P %d", plan->P));
        S(fmt("#define UVU_DX %d", plan->Dx));
        S(fmt("#define UVU_DY %d", plan->Dy));
        S(fmt("#define UVU_DO %d", plan->Do));
        S(fmt("#define RD_H %d", H));
        S(fmt("#define RD_NE %d", NE));
        S(fmt("#define RD_NG %d", split_n));
        S(fmt("#define RD_TPB %d", rw * 32));
        S(fmt("#define RD_RPB %d", rw));
        S(fmt("#define RD_NSL %d", A.radial_nsl));
        S("#define RD_WSM 1");
        S("#define RD_WSTR 32");
        S(fmt("#define RD_P2 %d", P2));
        S("#define RD_PACKED 1");
        S(fmt("#define RD_MINB %d", minb));
        S("__device__ unsigned int uvu_status_word;  // no bounded waits in this module: stays 0");
        G.emit_pair_helpers(S);
        G.radial_h_ = H;
        G.emit_fwd_radial(S, rg, NE, true, true);
        return S.o.str();
    }
    A.radial_gblk = 1;
    const int NG = int(rg.size());
    const size_t wsm_bytes = packed ? wsm_packed : wsm_plain;
    A.radial_wsm = packed || wsm_bytes <= 200 * 1024;
    const size_t smem = A.radial_wsm ? wsm_bytes : 0;
    const int fit = smem ? int(std::min<size_t>(4, (227 * 1024) / (smem + 1024))) : 4;
    int rw = NG * std::max(1, (fit == 1 ? 12 : 6) / NG);
    if (const char* e = std::getenv("UVU_RAD_RW")) rw = NG * std::max(1, std::atoi(e) / NG);
    rw = std::min(rw, NG * std::max(1, 32 / NG));
    if (rw * 32 > 1024) rw = NG;
    const int minb = std::max(1, std::min({fit, A.minb[0], 2048 / (rw * 32)}));
    A.minb_eff[0] = minb;
    A.radial_nsl = (plan->U + 31) / 32;
    A.radial_rpb = rw / NG;
    A.g[0] = {rw * 32, 1, smem, true};
    A.g[1] = {};
    Src S;
    S("// Generated by the UVU planner: forward with fused radial weights (last layer in registers).");
    S(fmt("// irreps_x=%s irreps_sh=%s lmax_out=%d dtype=%s hidden=%d", plan->irreps_x.c_str(), plan->irreps_sh.c_str(),
          plan->lmax_out, G.f64 ? "fp64" : "fp32", H));
    S(fmt("#define UVU_U %d", plan->U));
    S(fmt("#define UVU_P %d", plan->P));
    S(fmt("#define UVU_DX %d", plan->Dx));
    S(fmt("#define UVU_DY %d", plan->Dy));
    S(fmt("#define UVU_DO %d", plan->Do));
    S(fmt("#define RD_H %d", H));
    S(fmt("#define RD_NE %d", NE));
    S(fmt("#define RD_NG %d", NG));
    S(fmt("#define RD_TPB %d", rw * 32));
    S(fmt("#define RD_RPB %d", rw / NG));
    S(fmt("#define RD_NSL %d", A.radial_nsl));
    S(fmt("#define RD_WSM %d", A.radial_wsm ? 1 : 0));
    S(fmt("#define RD_WSTR %s", A.radial_wsm ? "32" : "UVU_U"));
    S(fmt("#define RD_P2 %d", P2));
    S(fmt("#define RD_PACKED %d", packed ? 1 : 0));
    S(fmt("#define RD_MINB %d", minb));
    S("__device__ unsigned int uvu_status_word;  // no bounded waits in this module: stays 0");
    G.emit_pair_helpers(S);
    G.radial_h_ = H;
    G.emit_fwd_radial(S, rg, NE, packed);
    return S.o.str();
}
}  // namespace

// Source of an auxiliary module: the double backward (AUX_HVP) or the batched tensor product
// with per-sample (AUX_TP) or batch-shared (AUX_TP_SHARED) weights.  For U >= 32 these are the
// pipelined receiver kernels in their dual-operand / single-edge-receiver variants; the double
// backward of smaller plans uses the direct-load kernels, and the batched tensor product needs
// the pipelined plan (the C ABI refuses it otherwise).
std::string emit_aux_source(Plan* plan, int kind) {
    if (kind == AUX_RADIAL) return emit_radial_source(plan);
    Gen G{plan, plan->dtype == UVU_F64, plan->dtype == UVU_F64 ? "double" : "float"};
    AuxBuild& A = plan->aux[kind];
    const int U = plan->U, NG = int(plan->groups.size()), UP = plan->U_pad;
    const int owner_threads = UP * NG;
    const int rpb = std::max(1, 128 / owner_threads);
    const int segw = std::min(UP, 32);
    const int segs = NG * ((UP + 31) / 32);
    const int ch = 16;
    const int ncw = NG * UP / 32;
    const bool pipe = plan->pipelined_recv;
    const bool ostage = !(std::getenv("UVU_PIPE_OSTAGE") && std::atoi(std::getenv("UVU_PIPE_OSTAGE")) == 0);
    const bool gstage = !(std::getenv("UVU_PIPE_GSTAGE") && std::atoi(std::getenv("UVU_PIPE_GSTAGE")) == 0);
    const bool hvp = kind == AUX_HVP, tp = !hvp, wsh = kind == AUX_TP_SHARED;
    Gen::RecvPipe RF, RE;
    if (pipe) {
        RF = G.fwd_pipe(ncw, A.minb[0], ostage, hvp, tp, wsh);
        RE = G.recv_pipe(true, ncw, false, 0, gstage, hvp, tp, wsh);
        // the double backward's edge kernel (one edge per stage, both operand sets) also takes a
        // third stage when it costs no resident block (MACE-medium: 1.63 -> 1.57 ms); the plain
        // edge kernels measured slower with one
        if (hvp && RE.ch == 1 && !std::getenv("UVU_PIPE_NST")) {
            const Gen::RecvPipe R3 = G.recv_pipe(true, ncw, false, 1, RE.gst, hvp, tp, wsh, 3);
            if (Gen::minb(R3.total) >= std::min(Gen::minb(RE.total), A.minb[1])) RE = R3;
        }
        A.g[0] = {ncw * 32 + 32, 1, RF.total, true};
        A.g[1] = {ncw * 32 + 32, 1, RE.total, true};
    } else {
        A.g[0] = {rpb * owner_threads, rpb, 0, false};
        A.g[1] = {rpb * owner_threads, rpb, size_t(rpb) * segs * ch * plan->Dy * plan->elem(), false};
    }
    Src S;
    S(fmt("// Generated by the UVU planner: %s of the channel-wise CG tensor product.",
          hvp ? "double backward (HVP) of the convolution" : wsh ? "batched product, batch-shared weights" : "batched product, per-sample weights"));
    S(fmt("// irreps_x=%s irreps_sh=%s lmax_out=%d dtype=%s", plan->irreps_x.c_str(), plan->irreps_sh.c_str(),
          plan->lmax_out, G.f64 ? "fp64" : "fp32"));
    S(fmt("#define UVU_U %d", U));
    S(fmt("#define UVU_UP %d", UP));
    S(fmt("#define UVU_P %d", plan->P));
    S(fmt("#define UVU_DX %d", plan->Dx));
    S(fmt("#define UVU_DY %d", plan->Dy));
    S(fmt("#define UVU_DO %d", plan->Do));
    S(fmt("#define UVU_G %d", NG));
    S(fmt("#define UVU_RPB %d", rpb));
    S(fmt("#define UVU_TPB %d", rpb * owner_threads));
    S(fmt("#define UVU_SEGW %d", segw));
    S(fmt("#define UVU_SEGS %d", segs));
    S(fmt("#define UVU_CH %d", ch));
    S(fmt("#define UVU_NCW %d", ncw));
    S(fmt("#define UVU_NCT %d", ncw * 32));
    S("__device__ __forceinline__ void block_sync() { asm volatile(\"barrier.sync 0;\" ::: \"memory\"); }");
    S("__device__ __forceinline__ void red_add_v4(float* a, float p, float q, float r, float s) {");
    S("  asm volatile(\"red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\" :: \"l\"(a), \"f\"(p), \"f\"(q), \"f\"(r), \"f\"(s) : \"memory\");");
    S("}");
    G.emit_pair_helpers(S);
    if (pipe) {
        G.emit_pipe_helpers(S);
        G.emit_recv_pipe_defines(S, RF, "FW", A.minb[0], A.minb_eff[0]);
        G.emit_recv_pipe_defines(S, RE, "EG", A.minb[1], A.minb_eff[1]);
        G.no_identity = hvp;
        G.emit_fwd_v2(S, RF);
        G.emit_edge_v2(S, RE);
        G.no_identity = false;
    } else if (hvp) {
        G.emit_hvp_kernels(S);
    }
    return S.o.str();
}

}  // namespace uvu
