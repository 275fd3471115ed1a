// Irreps parsing, path enumeration, layouts and register grouping for a plan.
//
// Paths: for each x irrep (string order), each SH irrep (string order) and each l3 ascending over
// |l1-l2| .. min(l1+l2, lmax_out), one path with output parity p1*p2 ("all parity-allowed
// channel-wise paths": every triangle-allowed l3 is kept).  Channel-wise (UVU) structure: every
// x irrep carries the same multiplicity U and the SH irreps multiplicity 1, so each
// (receiver, channel) owner of "Receiver-streaming convolutions for channel-wise UVU tensor
// products" (opening post, ownership paragraph) sees one scalar weight per path.
#include <cctype>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "plan.h"

namespace uvu {

namespace {
constexpr int kMaxLIn = 4;
constexpr int kMaxLOut = 8;
}  // namespace

bool parse_irreps(const char* s, std::vector<Irrep>* out, std::string* err) {
    out->clear();
    if (!s || !*s) {
        *err = "empty irreps string";
        return false;
    }
    const char* p = s;
    while (true) {
        while (*p == ' ') ++p;
        if (!std::isdigit((unsigned char)*p)) {
            *err = std::string("expected multiplicity in irreps '") + s + "'";
            return false;
        }
        char* end = nullptr;
        long mul = std::strtol(p, &end, 10);
        p = end;
        if (*p != 'x') {
            *err = std::string("expected 'x' in irreps '") + s + "'";
            return false;
        }
        ++p;
        if (!std::isdigit((unsigned char)*p)) {
            *err = std::string("expected l in irreps '") + s + "'";
            return false;
        }
        long l = std::strtol(p, &end, 10);
        p = end;
        int par;
        if (*p == 'e') par = 1;
        else if (*p == 'o') par = -1;
        else {
            *err = std::string("expected parity e/o in irreps '") + s + "'";
            return false;
        }
        ++p;
        if (mul <= 0 || mul > 4096 || l < 0 || l > 64) {
            *err = std::string("multiplicity or l out of range in '") + s + "'";
            return false;
        }
        out->push_back({int(mul), int(l), par});
        while (*p == ' ') ++p;
        if (*p == '\0') break;
        if (*p != '+') {
            *err = std::string("expected '+' in irreps '") + s + "'";
            return false;
        }
        ++p;
    }
    return true;
}

uvu_status build_paths(Plan* plan, std::string* err) {
    if (!parse_irreps(plan->irreps_x.c_str(), &plan->xs, err)) return UVU_ERR_INVALID_ARGUMENT;
    if (!parse_irreps(plan->irreps_sh.c_str(), &plan->ys, err)) return UVU_ERR_INVALID_ARGUMENT;
    const int U = plan->xs[0].mul;
    for (size_t i = 0; i < plan->xs.size(); ++i) {
        if (plan->xs[i].mul != U) {
            *err = "channel-wise (UVU) plan needs one multiplicity for every x irrep";
            return UVU_ERR_INVALID_ARGUMENT;
        }
        for (size_t j = 0; j < i; ++j)
            if (plan->xs[j].l == plan->xs[i].l) {
                *err = "each l may appear once in irreps_x";
                return UVU_ERR_INVALID_ARGUMENT;
            }
        if (plan->xs[i].l > kMaxLIn) {
            *err = "irreps_x: l > 4 is not supported";
            return UVU_ERR_UNSUPPORTED;
        }
    }
    for (const Irrep& y : plan->ys) {
        if (y.mul != 1) {
            *err = "irreps_sh terms must have multiplicity 1";
            return UVU_ERR_INVALID_ARGUMENT;
        }
        if (y.l > kMaxLIn) {
            *err = "irreps_sh: l > 4 is not supported";
            return UVU_ERR_UNSUPPORTED;
        }
    }
    if (plan->lmax_out < 0 || plan->lmax_out > kMaxLOut) {
        *err = "lmax_out must be in [0, 8]";
        return UVU_ERR_INVALID_ARGUMENT;
    }
    plan->U = U;
    plan->paths.clear();
    int xoff = 0, ooff = 0;
    for (size_t ix = 0; ix < plan->xs.size(); ++ix) {
        const Irrep& a = plan->xs[ix];
        int yoff = 0;
        for (size_t iy = 0; iy < plan->ys.size(); ++iy) {
            const Irrep& b = plan->ys[iy];
            const int lo = std::abs(a.l - b.l);
            const int hi = std::min(a.l + b.l, plan->lmax_out);
            for (int l3 = lo; l3 <= hi; ++l3) {
                PathInfo p;
                p.l1 = a.l;
                p.l2 = b.l;
                p.l3 = l3;
                p.parity = a.parity * b.parity;
                p.ix = int(ix);
                p.iy = int(iy);
                p.xoff = xoff;
                p.yoff = yoff;
                p.ooff = ooff;
                p.cg = real_cg_dense(a.l, b.l, l3);
                const int d2 = 2 * b.l + 1, d3 = 2 * l3 + 1;
                for (size_t i = 0; i < p.cg.size(); ++i) {
                    if (std::abs(p.cg[i]) > 1e-12) {
                        const int m1 = int(i / (size_t(d2) * d3));
                        const int m2 = int((i / d3) % d2);
                        const int m3 = int(i % d3);
                        p.nz.push_back({m1, m2, m3, p.cg[i]});
                    }
                }
                ooff += d3;
                plan->paths.push_back(std::move(p));
            }
            yoff += 2 * b.l + 1;
        }
        xoff += 2 * a.l + 1;
    }
    plan->Dx = xoff;
    plan->Do = ooff;
    plan->Dy = 0;
    for (const Irrep& b : plan->ys) plan->Dy += 2 * b.l + 1;
    plan->P = int(plan->paths.size());
    if (plan->P == 0) {
        *err = "no path satisfies the triangle rule with l3 <= lmax_out";
        return UVU_ERR_UNSUPPORTED;
    }
    // Register groups: consecutive paths whose output width fits one thread's accumulator
    // budget.  A (receiver, channel) owner is split into one thread per group when the whole
    // output row would not fit in registers (fp64, wide l).
    // Below 32 channels one warp spans several owners, so a single group keeps every warp on one
    // code path (the dY shuffles need that).
    const int budget = U < 32 ? (1 << 30) : (plan->dtype == UVU_F64 ? 40 : 112);
    plan->groups.clear();
    std::vector<int> cur;
    int width = 0;
    for (int p = 0; p < plan->P; ++p) {
        const int d3 = 2 * plan->paths[p].l3 + 1;
        if (!cur.empty() && width + d3 > budget) {
            plan->groups.push_back(cur);
            cur.clear();
            width = 0;
        }
        cur.push_back(p);
        width += d3;
    }
    plan->groups.push_back(cur);
    return UVU_OK;
}

}  // namespace uvu
