// planner.cpp -- host-side planner: irreps parsing, path enumeration, CG blocks
// from Racah's closed form, real basis, and the per-plan kernel tables.
//
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
// Abstract (static analysis at model compile time) and Figures 1-2 (the
// coefficient tensor is block-sparse, one block per (l1, l2, l3), each block
// itself sparse).  The pages print no formula; the coefficients follow the
// standard closed form of Racah with the Condon-Shortley phase.
//
// Exactness: the alternating Racah sum is accumulated as an exact integer
// (each term times (j1+j2+J)! is a multinomial coefficient), and the square
// root of the prefactor is assembled from prime exponents, so the only
// roundings are a handful of final double operations.  Compile with
// -ffp-contract=off so x86-64 and aarch64 hosts give identical tables.
#include <algorithm>
#include <cctype>
#include <cmath>
#include <complex>
#include <cstring>
#include <numeric>

#include "internal.h"

namespace cgtp {

namespace {
thread_local std::string g_last_error;
}

cgtp_status fail(cgtp_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}
void clear_error() { g_last_error.clear(); }
const char* last_error_cstr() { return g_last_error.c_str(); }

// ---------------------------------------------------------------------------
// irreps strings
// ---------------------------------------------------------------------------
bool parse_irreps(const char* s, std::vector<Irrep>* out, std::string* err) {
  out->clear();
  if (!s) {
    *err = "null irreps string";
    return false;
  }
  std::string str;
  for (const char* c = s; *c; ++c)
    if (!std::isspace(static_cast<unsigned char>(*c))) str.push_back(*c);
  if (str.empty()) {
    *err = "empty irreps string";
    return false;
  }
  size_t pos = 0;
  while (pos <= str.size()) {
    size_t next = str.find('+', pos);
    if (next == std::string::npos) next = str.size();
    std::string term = str.substr(pos, next - pos);
    if (term.empty()) {
      *err = "empty term in irreps '" + std::string(s) + "'";
      return false;
    }
    long mul = 1;
    size_t x = term.find('x');
    std::string ir = term;
    if (x != std::string::npos) {
      std::string m = term.substr(0, x);
      if (m.empty() || !std::all_of(m.begin(), m.end(), ::isdigit) || m.size() > 6) {
        *err = "bad multiplicity in '" + term + "'";
        return false;
      }
      mul = std::stol(m);
      ir = term.substr(x + 1);
    }
    if (ir.size() < 2 || (ir.back() != 'e' && ir.back() != 'o')) {
      *err = "bad irrep '" + term + "' (expected like 8x1o)";
      return false;
    }
    std::string ls = ir.substr(0, ir.size() - 1);
    if (!std::all_of(ls.begin(), ls.end(), ::isdigit) || ls.size() > 3) {
      *err = "bad l in '" + term + "'";
      return false;
    }
    int l = std::stoi(ls);
    if (l > kMaxL) {
      *err = "l = " + ls + " exceeds the supported maximum 7";
      return false;
    }
    if (mul < 1 || mul > 65536) {
      *err = "multiplicity out of range in '" + term + "'";
      return false;
    }
    out->push_back({static_cast<int>(mul), l, ir.back() == 'e' ? 1 : -1});
    pos = next + 1;
    if (next == str.size()) break;
  }
  return true;
}

// ---------------------------------------------------------------------------
// Clebsch-Gordan coefficients (Racah), exact sum
// ---------------------------------------------------------------------------
namespace {
const int kPrimes[] = {2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37, 41, 43, 47};
constexpr int kNP = sizeof(kPrimes) / sizeof(int);

void add_int(int* e, int n, int sign) {  // exponents of n
  for (int i = 0; i < kNP && n > 1; ++i)
    while (n % kPrimes[i] == 0) {
      e[i] += sign;
      n /= kPrimes[i];
    }
}
void add_fact(int* e, int n, int sign) {
  for (int k = 2; k <= n; ++k) add_int(e, k, sign);
}
unsigned __int128 ufact(int n) {
  unsigned __int128 r = 1;
  for (int k = 2; k <= n; ++k) r *= static_cast<unsigned>(k);
  return r;
}
}  // namespace

double cg_complex(int j1, int m1, int j2, int m2, int J, int M) {
  if (m1 + m2 != M) return 0.0;
  if (J < std::abs(j1 - j2) || J > j1 + j2) return 0.0;
  if (std::abs(m1) > j1 || std::abs(m2) > j2 || std::abs(M) > J) return 0.0;
  const int F = j1 + j2 + J;
  // sum_k (-1)^k F! / (k! (j1+j2-J-k)! (j1-m1-k)! (j2+m2-k)! (J-j2+m1+k)! (J-j1-m2+k)!)
  __int128 S = 0;
  const unsigned __int128 Ff = ufact(F);
  for (int k = 0; k <= j1 + j2 - J; ++k) {
    int d[6] = {k, j1 + j2 - J - k, j1 - m1 - k, j2 + m2 - k, J - j2 + m1 + k, J - j1 - m2 + k};
    bool ok = true;
    for (int v : d) ok &= (v >= 0);
    if (!ok) continue;
    unsigned __int128 t = Ff;
    for (int v : d) t /= ufact(v);  // each partial quotient is an integer (multinomial)
    S += (k & 1) ? -static_cast<__int128>(t) : static_cast<__int128>(t);
  }
  if (S == 0) return 0.0;
  // CG^2 = S^2 * (2J+1) (J+j1-j2)! (J-j1+j2)! (j1+j2-J)! (J+M)! (J-M)! (j1-m1)! (j1+m1)!
  //        (j2-m2)! (j2+m2)! / ((j1+j2+J+1)! * F!^2)
  int e[kNP] = {0};
  add_int(e, 2 * J + 1, +1);
  add_fact(e, J + j1 - j2, +1);
  add_fact(e, J - j1 + j2, +1);
  add_fact(e, j1 + j2 - J, +1);
  add_fact(e, J + M, +1);
  add_fact(e, J - M, +1);
  add_fact(e, j1 - m1, +1);
  add_fact(e, j1 + m1, +1);
  add_fact(e, j2 - m2, +1);
  add_fact(e, j2 + m2, +1);
  add_fact(e, F + 1, -1);
  add_fact(e, F, -2);
  unsigned __int128 num = 1, den = 1;
  unsigned long long rad = 1;
  for (int i = 0; i < kNP; ++i) {
    int q = e[i] >= 0 ? e[i] / 2 : -((-e[i] + 1) / 2);  // floor(e/2)
    int r = e[i] - 2 * q;                               // 0 or 1
    for (int t = 0; t < q; ++t) num *= static_cast<unsigned>(kPrimes[i]);
    for (int t = 0; t < -q; ++t) den *= static_cast<unsigned>(kPrimes[i]);
    if (r) rad *= static_cast<unsigned>(kPrimes[i]);
  }
  const double sabs = static_cast<double>(S < 0 ? -S : S);
  double v = sabs * (static_cast<double>(num) / static_cast<double>(den)) *
             std::sqrt(static_cast<double>(rad));
  return S < 0 ? -v : v;
}

// ---------------------------------------------------------------------------
// real basis and the real, component-normalised block
// ---------------------------------------------------------------------------
namespace {
using cd = std::complex<double>;

// Row a (real m = a - l) of the complex -> real change of basis, as at most two
// (column, value) pairs.  m>0: (Y^{-m} + (-1)^m Y^m)/sqrt2; m=0: Y^0;
// m<0: i (Y^m - (-1)^m Y^{-m})/sqrt2.
int real_row(int l, int a, int* cols, cd* vals) {
  const int m = a - l;
  const double r = 1.0 / std::sqrt(2.0);
  if (m == 0) {
    cols[0] = l;
    vals[0] = 1.0;
    return 1;
  }
  const double sgn = ((m < 0 ? -m : m) % 2) ? -1.0 : 1.0;  // (-1)^m
  if (m > 0) {
    cols[0] = -m + l;
    vals[0] = r;
    cols[1] = m + l;
    vals[1] = sgn * r;
  } else {
    cols[0] = m + l;
    vals[0] = cd(0.0, r);
    cols[1] = -m + l;
    vals[1] = cd(0.0, -sgn * r);
  }
  return 2;
}
}  // namespace

std::vector<double> real_cg_block(int l1, int l2, int l3) {
  const int D1 = 2 * l1 + 1, D2 = 2 * l2 + 1, D3 = 2 * l3 + 1;
  std::vector<double> out(static_cast<size_t>(D1) * D2 * D3, 0.0);
  if (l3 < std::abs(l1 - l2) || l3 > l1 + l2) return out;
  std::vector<cd> T(out.size());
  int c1[2], c2[2], c3[2];
  cd v1[2], v2[2], v3[2];
  for (int a = 0; a < D1; ++a) {
    int n1 = real_row(l1, a, c1, v1);
    for (int b = 0; b < D2; ++b) {
      int n2 = real_row(l2, b, c2, v2);
      for (int c = 0; c < D3; ++c) {
        int n3 = real_row(l3, c, c3, v3);
        cd acc = 0.0;
        for (int i = 0; i < n1; ++i)
          for (int j = 0; j < n2; ++j)
            for (int k = 0; k < n3; ++k) {
              const double cg = cg_complex(l1, c1[i] - l1, l2, c2[j] - l2, l3, c3[k] - l3);
              if (cg != 0.0) acc += v1[i] * v2[j] * std::conj(v3[k]) * cg;
            }
        T[(static_cast<size_t>(a) * D2 + b) * D3 + c] = acc;
      }
    }
  }
  double re = 0, im = 0;
  for (const cd& t : T) {
    re = std::max(re, std::abs(t.real()));
    im = std::max(im, std::abs(t.imag()));
  }
  const bool use_re = re >= im;
  double norm2 = 0;
  for (size_t i = 0; i < T.size(); ++i) {
    out[i] = use_re ? T[i].real() : T[i].imag();
    norm2 += out[i] * out[i];
  }
  const double inv = 1.0 / std::sqrt(norm2);
  size_t first = 0;
  while (first < out.size() && std::abs(out[first] * inv) <= 1e-12) ++first;
  const double sign = (out[first] < 0) ? -1.0 : 1.0;
  const double scale = sign * inv;
  const double comp = std::sqrt(static_cast<double>(D3));
  for (double& v : out) {
    v *= scale;
    v = (std::abs(v) > 1e-13) ? v * comp : 0.0;
  }
  return out;
}

// ---------------------------------------------------------------------------
// paths
// ---------------------------------------------------------------------------
static std::vector<int> offsets(const std::vector<Irrep>& irr) {
  std::vector<int> o;
  int acc = 0;
  for (const auto& i : irr) {
    o.push_back(acc);
    acc += i.mul * (2 * i.l + 1);
  }
  return o;
}
static int64_t dim(const std::vector<Irrep>& irr) {
  int64_t d = 0;
  for (const auto& i : irr) d += static_cast<int64_t>(i.mul) * (2 * i.l + 1);
  return d;
}

cgtp_status build_paths(cgtp_plan_s* plan, const cgtp_instr* instr, int n_instr) {
  std::vector<cgtp_instr> list;
  if (instr && n_instr > 0) {
    list.assign(instr, instr + n_instr);
  } else {
    for (int i1 = 0; i1 < static_cast<int>(plan->in1.size()); ++i1)
      for (int i2 = 0; i2 < static_cast<int>(plan->in2.size()); ++i2) {
        const Irrep a = plan->in1[i1], b = plan->in2[i2];
        for (int l3 = std::abs(a.l - b.l); l3 <= a.l + b.l; ++l3) {
          const int p3 = a.p * b.p;
          for (int io = 0; io < static_cast<int>(plan->out.size()); ++io)
            if (plan->out[io].l == l3 && plan->out[io].p == p3) {
              list.push_back({i1, i2, io});
              break;
            }
        }
      }
  }
  if (list.empty()) return fail(CGTP_EINVAL, "the plan has no path");
  const auto o1 = offsets(plan->in1), o2 = offsets(plan->in2), oo = offsets(plan->out);
  int64_t ooff = 0, woff = 0;
  std::vector<Irrep> derived;
  for (const auto& ins : list) {
    if (ins.i_in1 < 0 || ins.i_in1 >= static_cast<int>(plan->in1.size()) || ins.i_in2 < 0 ||
        ins.i_in2 >= static_cast<int>(plan->in2.size()) || ins.i_out < 0 ||
        ins.i_out >= static_cast<int>(plan->out.size()))
      return fail(CGTP_EINVAL, "instruction index out of range");
    const Irrep a = plan->in1[ins.i_in1], b = plan->in2[ins.i_in2], c = plan->out[ins.i_out];
    if (c.l < std::abs(a.l - b.l) || c.l > a.l + b.l)
      return fail(CGTP_EINVAL, "instruction violates the triangle rule");
    if (c.p != a.p * b.p) return fail(CGTP_EINVAL, "instruction violates parity");
    PathHost p;
    p.i1 = ins.i_in1;
    p.i2 = ins.i_in2;
    p.io = ins.i_out;
    p.l1 = a.l;
    p.l2 = b.l;
    p.l3 = c.l;
    p.mul1 = a.mul;
    p.off1 = o1[ins.i_in1];
    p.off2 = o2[ins.i_in2];
    if (plan->mode == CGTP_UVU) {
      p.mul_out = a.mul;
      p.ooff = static_cast<int>(ooff);
      p.woff = static_cast<int>(woff);
      ooff += static_cast<int64_t>(a.mul) * (2 * c.l + 1);
      woff += a.mul;
      derived.push_back({a.mul, c.l, c.p});
    } else {
      p.mul_out = c.mul;
      p.ooff = oo[ins.i_out];
      p.woff = static_cast<int>(woff);
      woff += static_cast<int64_t>(a.mul) * c.mul;
    }
    p.C = real_cg_block(p.l1, p.l2, p.l3);
    plan->paths.push_back(std::move(p));
  }
  if (plan->mode == CGTP_UVU) plan->out = derived;
  plan->d1 = dim(plan->in1);
  plan->d2 = dim(plan->in2);
  plan->d_out = dim(plan->out);
  plan->w_numel = woff;
  if (plan->d1 > (1 << 24) || plan->d_out > (1 << 24) || plan->w_numel > (1 << 26))
    return fail(CGTP_EUNSUPPORTED, "feature dimensions too large");
  return CGTP_OK;
}

// ---------------------------------------------------------------------------
// layouts: groups of paths, coefficient term lists, per-warp work items
// ---------------------------------------------------------------------------
static int pad_to(int v, int q) { return (v + q - 1) / q * q; }

cgtp_status build_layout(const cgtp_plan_s* plan, int chunk, size_t budget, LayoutHost* L) {
  const size_t es = plan->dtype == CGTP_F64 ? 8 : 4;
  const int vec = plan->dtype == CGTP_F64 ? 2 : 4;  // elements per 16-byte vector
  const int P = static_cast<int>(plan->paths.size());
  const int d2p = pad_to(static_cast<int>(plan->d2), vec);
  L->chunk = chunk;
  L->groups.clear();
  // Greedy grouping of consecutive paths under the shared-memory budget of
  // both kernels (forward: Y chunk + cy + out slice; backward: x row + Y chunk
  // + cy + gc partials + gx partials).
  auto smem_of = [&](int p0, int p1, size_t* fwd, size_t* bwd) {
    int cy = 0, dog = 0, gxp = 0, nub = 1;
    for (int p = p0; p < p1; ++p) {
      const auto& q = plan->paths[p];
      const int D1 = 2 * q.l1 + 1, D3 = 2 * q.l3 + 1;
      cy += pad_to(D1 * D3, vec);
      dog += q.mul1 * D3;
      gxp += q.mul1 * D1;
      nub = std::max(nub, (q.mul1 + 31) / 32);
    }
    const size_t ints = 16 * static_cast<size_t>(chunk);
    *fwd = es * (static_cast<size_t>(chunk) * (d2p + cy) + pad_to(dog, vec)) + ints;
    *bwd = es * (pad_to(static_cast<int>(plan->d1), vec) + static_cast<size_t>(chunk) * d2p +
                 static_cast<size_t>(chunk) * cy * (1 + nub) + pad_to(gxp, vec)) +
           ints;
  };
  int p0 = 0;
  while (p0 < P) {
    int p1 = p0 + 1;
    size_t f, b;
    smem_of(p0, p1, &f, &b);
    if (f > budget || b > budget)
      return fail(CGTP_EUNSUPPORTED, "a single path does not fit in shared memory");
    while (p1 < P) {
      smem_of(p0, p1 + 1, &f, &b);
      if (f > budget || b > budget) break;
      ++p1;
    }
    GroupDev g{};
    g.p0 = p0;
    g.p1 = p1;
    L->groups.push_back(g);
    p0 = p1;
  }
  L->cy_begin.clear();
  L->cy_col.clear();
  L->cy_coef.clear();
  L->gy_begin.clear();
  L->gy_slot.clear();
  L->gy_nub.clear();
  L->gy_coef.clear();
  L->item_begin.clear();
  L->items.clear();
  L->gx_begin.clear();
  L->gx_paths.clear();
  L->smem_fwd = L->smem_bwd = 0;
  const int n_in1 = static_cast<int>(plan->in1.size());
  L->in1_off = offsets(plan->in1);
  L->in1_off.push_back(static_cast<int>(plan->d1));
  L->paths.assign(P, PathDev{});
  for (int p = 0; p < P; ++p) {
    const auto& q = plan->paths[p];
    PathDev& d = L->paths[p];
    d.l1 = q.l1;
    d.l2 = q.l2;
    d.l3 = q.l3;
    d.D1 = 2 * q.l1 + 1;
    d.D2 = 2 * q.l2 + 1;
    d.D3 = 2 * q.l3 + 1;
    d.mul = q.mul1;
    d.mul_out = q.mul_out;
    d.off1 = q.off1;
    d.off2 = q.off2;
    d.ooff = q.ooff;
    d.woff = q.woff;
    d.i1 = q.i1;
  }
  for (auto& g : L->groups) {
    const auto& first = plan->paths[g.p0];
    const auto& last = plan->paths[g.p1 - 1];
    g.o0 = first.ooff;
    g.o1 = last.ooff + last.mul1 * (2 * last.l3 + 1);
    g.w0 = first.woff;
    g.w1 = last.woff + last.mul1;
    // cy layout: per path a dense [D1][D3] block padded to a 16-byte multiple
    std::vector<int> cyoff(g.p1 - g.p0), gxoff(g.p1 - g.p0);
    int cy = 0, gxp = 0, nub = 1;
    for (int p = g.p0; p < g.p1; ++p) {
      const auto& q = plan->paths[p];
      cyoff[p - g.p0] = cy;
      gxoff[p - g.p0] = gxp;
      cy += pad_to((2 * q.l1 + 1) * (2 * q.l3 + 1), vec);
      gxp += q.mul1 * (2 * q.l1 + 1);
      nub = std::max(nub, (q.mul1 + 31) / 32);
    }
    g.cy_size = cy;
    g.gxp_size = gxp;
    for (int p = g.p0; p < g.p1; ++p) {
      PathDev& d = L->paths[p];
      d.ooff_g = d.ooff - g.o0;
      d.woff_g = d.woff - g.w0;
      d.cyoff_g = cyoff[p - g.p0];
      d.gxpoff_g = gxoff[p - g.p0];
    }
    g.nub = nub;
    // forward terms: cy[slot] = sum coef * Y[col]
    g.cy_base = static_cast<int>(L->cy_begin.size());
    std::vector<std::vector<std::pair<int, double>>> slot_terms(cy);
    // backward terms: gY[c] = sum coef * gc[slot] (summed over channel blocks)
    std::vector<std::vector<std::pair<int, double>>> col_terms(plan->d2);
    std::vector<std::vector<int>> col_nub(plan->d2);
    for (int p = g.p0; p < g.p1; ++p) {
      const auto& q = plan->paths[p];
      const int D1 = 2 * q.l1 + 1, D2 = 2 * q.l2 + 1, D3 = 2 * q.l3 + 1;
      for (int m1 = 0; m1 < D1; ++m1)
        for (int m2 = 0; m2 < D2; ++m2)
          for (int m3 = 0; m3 < D3; ++m3) {
            const double c = q.C[(static_cast<size_t>(m1) * D2 + m2) * D3 + m3];
            if (c == 0.0) continue;
            const int slot = cyoff[p - g.p0] + m1 * D3 + m3;
            slot_terms[slot].push_back({q.off2 + m2, c});
            col_terms[q.off2 + m2].push_back({slot, c});
            col_nub[q.off2 + m2].push_back((q.mul1 + 31) / 32);
          }
    }
    for (int s = 0; s < cy; ++s) {
      L->cy_begin.push_back(static_cast<int>(L->cy_col.size()));
      for (auto& t : slot_terms[s]) {
        L->cy_col.push_back(t.first);
        L->cy_coef.push_back(t.second);
      }
    }
    L->cy_begin.push_back(static_cast<int>(L->cy_col.size()));
    g.gy_base = static_cast<int>(L->gy_begin.size());
    for (int c = 0; c < plan->d2; ++c) {
      L->gy_begin.push_back(static_cast<int>(L->gy_slot.size()));
      for (size_t t = 0; t < col_terms[c].size(); ++t) {
        L->gy_slot.push_back(col_terms[c][t].first);
        L->gy_coef.push_back(col_terms[c][t].second);
        L->gy_nub.push_back(col_nub[c][t]);
      }
    }
    L->gy_begin.push_back(static_cast<int>(L->gy_slot.size()));
    // work items: (path, 32-channel block), longest first onto the least loaded warp
    struct It {
      int path, u0;
      double cost;
    };
    std::vector<It> its;
    for (int p = g.p0; p < g.p1; ++p) {
      const auto& q = plan->paths[p];
      const int D1 = 2 * q.l1 + 1, D3 = 2 * q.l3 + 1;
      for (int u0 = 0; u0 < q.mul1; u0 += 32)
        its.push_back({p, u0, static_cast<double>(D1 * D3 + D1 + D3 + 4)});
    }
    std::stable_sort(its.begin(), its.end(), [](const It& a, const It& b) { return a.cost > b.cost; });
    std::vector<std::vector<Item>> per_warp(kWarps);
    std::vector<double> load(kWarps, 0.0);
    for (const auto& it : its) {
      const int w = static_cast<int>(std::min_element(load.begin(), load.end()) - load.begin());
      per_warp[w].push_back({it.path, it.u0});
      load[w] += it.cost;
    }
    g.item_base = static_cast<int>(L->item_begin.size());
    for (int w = 0; w < kWarps; ++w) {
      L->item_begin.push_back(static_cast<int>(L->items.size()));
      for (auto& i : per_warp[w]) L->items.push_back(i);
    }
    L->item_begin.push_back(static_cast<int>(L->items.size()));
    // gx reduction lists: for every in1 block, the group's paths reading it
    g.gx_base = static_cast<int>(L->gx_begin.size());
    for (int i1 = 0; i1 < n_in1; ++i1) {
      L->gx_begin.push_back(static_cast<int>(L->gx_paths.size()));
      for (int p = g.p0; p < g.p1; ++p)
        if (plan->paths[p].i1 == i1) L->gx_paths.push_back(p);
    }
    L->gx_begin.push_back(static_cast<int>(L->gx_paths.size()));
    size_t f, b;
    smem_of(g.p0, g.p1, &f, &b);
    L->smem_fwd = std::max(L->smem_fwd, f);
    L->smem_bwd = std::max(L->smem_bwd, b);
    // two-term form of the same cy terms
    L->cy2_base.push_back(static_cast<int>(L->cy2_col.size() / 2));
    for (int sl = 0; sl < cy; ++sl) {
      const auto& ts = slot_terms[sl];
      if (ts.size() > 2) return fail(CGTP_EUNSUPPORTED, "a cy slot has more than two CG terms");
      for (int k = 0; k < 2; ++k) {
        L->cy2_col.push_back(k < static_cast<int>(ts.size()) ? ts[k].first : 0);
        L->cy2_coef.push_back(k < static_cast<int>(ts.size()) ? ts[k].second : 0.0);
      }
    }
  }
  // pipelined forward kernel: [acc | 2 x (x rows, W rows, Y rows, src) | cy pairs]
  {
    int dog = 0, wg = 0, cy = 0;
    for (const auto& g : L->groups) {
      dog = std::max(dog, g.o1 - g.o0);
      wg = std::max(wg, g.w1 - g.w0);
      cy = std::max(cy, g.cy_size);
    }
    const int d1p = pad_to(static_cast<int>(plan->d1), vec);
    auto fwd2 = [&](int ch) {
      return es * (static_cast<size_t>(pad_to(dog, vec)) +
                   2 * static_cast<size_t>(ch) * (d1p + pad_to(wg, vec) + d2p) +
                   static_cast<size_t>(ch) * cy) + 2 * 4 * static_cast<size_t>(ch) + 64;
    };
    L->chunk2 = 0;
    for (int ch : {8, 4, 2})            // two CTAs per SM if possible
      if (fwd2(ch) <= 110 * 1024) { L->chunk2 = ch; break; }
    if (!L->chunk2)
      for (int ch : {8, 4, 2})          // else one CTA per SM
        if (fwd2(ch) <= 220 * 1024) { L->chunk2 = ch; break; }
    L->smem_fwd2 = L->chunk2 ? fwd2(L->chunk2) : 0;
  }
  return CGTP_OK;
}

}  // namespace cgtp
