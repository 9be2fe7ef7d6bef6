// Engram gate oracle: plain, slow, fp64 CPU definitions of what the GPU path
// computes.  THIS IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and
// the benchmark's CPU-baseline leg may load it; the product path never does.
// It shares no code, header or constant generator with the CUDA sources.
//
// Sources (web pages, cited by title and section):
//   [cuDNN-EG]  cuDNN Frontend, "Engram saved-state gate": semantics paragraph
//               (normalise X and key separately, FP32 reduce of X*weight*key,
//               signed square root with a 1e-6 clamp, sigmoid, out = X +
//               gate*shared_value rounded once to BF16, false mask -> X, eps
//               1e-20); layout paragraph (packed KV, backward writes the sum of
//               the four shared-value contributions); saved-state paragraph
//               ((gate, dot, rstd_X, rstd_key) per stream).
//   [TK-tests]  tile-kernels 1.0.0 sdist, tests/engram/test_engram_gate_fwd.py
//               and test_engram_gate_bwd.py (eps 1e-20, clamp 1e-6, grad_w is
//               a sum of partials, product rule for the two q/k weights).
//   [TileOPs]   TileOPs "Engram Operators", GateConv section:
//               EngramGateConvFwdOp (RMSNorm gating -> causal depthwise conv1d
//               with 4 taps -> SiLU + residual; saves vhat, alpha, rrms_h,
//               rrms_k, rrms_v) and EngramGateConvBwdOp (dH, dk, dv and fp32
//               drms_w_h, drms_w_v, dconv_w).
//
// Readings where the pages leave a step open are listed beside each function.
// Every function takes and returns fp64 arrays; conversion to and from bf16 is
// done by the separate oracle_bf16_* helpers below, so that the arithmetic of
// each op is a single fp64 evaluation followed by one rounding.
//
// Build: g++ -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }

// sign(0) = 0, as the signed square root of zero is zero.
double sgn(double a) { return a > 0.0 ? 1.0 : (a < 0.0 ? -1.0 : 0.0); }

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// bf16 helpers (the oracle's own; bf16 = 1 sign, 8 exponent, 7 mantissa bits)
// ---------------------------------------------------------------------------

// Exact widening of bf16 bit patterns to fp64.
void oracle_bf16_to_f64(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t bits = static_cast<uint32_t>(in[i]) << 16;
        float f;
        std::memcpy(&f, &bits, 4);
        out[i] = static_cast<double>(f);
    }
}

// One round-to-nearest-even step from fp64 straight to bf16 (no intermediate
// fp32 rounding).  NaN keeps its sign and becomes the canonical quiet NaN;
// values at or beyond the overflow threshold become infinity; values below
// the normal range go to bf16 subnormals (quantum 2^-133).
uint16_t oracle_round_bf16_one(double v) {
    uint16_t sign = std::signbit(v) ? 0x8000u : 0u;
    if (std::isnan(v)) return static_cast<uint16_t>(sign | 0x7FC0u);
    double a = std::fabs(v);
    if (std::isinf(a)) return static_cast<uint16_t>(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    std::frexp(a, &e);          // a in [2^(e-1), 2^e)
    int E = e - 1;              // a in [2^E, 2^(E+1))
    // quantum of the bf16 grid around a: 7 stored mantissa bits for normals,
    // a fixed 2^-133 step below 2^-126
    double q = (E < -126) ? std::ldexp(1.0, -133) : std::ldexp(1.0, E - 7);
    double m = a / q;                 // exact: q is a power of two
    double r = std::nearbyint(m);     // default mode: ties to even
    double res = r * q;               // exact
    if (res >= std::ldexp(1.0, 128)) return static_cast<uint16_t>(sign | 0x7F80u);
    float f = static_cast<float>(res);  // exact: res lies on the bf16 grid
    uint32_t bits;
    std::memcpy(&bits, &f, 4);
    return static_cast<uint16_t>(sign | ((bits >> 16) & 0x7FFFu));
}

void oracle_f64_to_bf16(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16_one(in[i]);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

// ---------------------------------------------------------------------------
// Saved-state gate, forward  ([cuDNN-EG] semantics + saved-state paragraphs)
//
//   x    (N, S, d)        stream s of token n
//   kv   (N, (S+1)*d)     keys for s = 0..S-1, then the shared value
//   w    (S, d)           fused fp32 weight (product of the q/k norm weights)
//   mask (N) or NULL      nonzero = true; NULL means all true
//   out  (N, S, d)        exact fp64 value of X + gate*v (rounded by caller)
//   saved (N, S, 4)       gate, dot, rstd_X, rstd_key
//
// Readings: "normalise" is RMS normalisation, rstd = 1/sqrt(mean(x^2)+eps),
// with no scale inside (the scales live in w); dot carries no temperature;
// the signed square root is sign(dot)*sqrt(max(|dot|, clamp)) with sign(0)=0;
// for a false mask the output is X and the stored gate is 0 while dot and
// both rstd are computed as usual, so that the backward (which takes no mask)
// sees a zero gate.
// ---------------------------------------------------------------------------
int oracle_gate_fwd(const double* x, const double* kv, const double* w,
                    const uint8_t* mask, int64_t N, int64_t S, int64_t d,
                    double eps, double clamp, double* out, double* saved) {
    if (N < 0 || S < 1 || d < 1) return 1;
    const int64_t kvw = (S + 1) * d;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        std::vector<double> xh(d), kh(d);
        const double* v = kv + n * kvw + S * d;
        const bool on = (mask == nullptr) || (mask[n] != 0);
        for (int64_t s = 0; s < S; ++s) {
            const double* xs = x + (n * S + s) * d;
            const double* ks = kv + n * kvw + s * d;
            const double* ws = w + s * d;
            double ssx = 0.0, ssk = 0.0;
            for (int64_t i = 0; i < d; ++i) {
                ssx += xs[i] * xs[i];
                ssk += ks[i] * ks[i];
            }
            const double rstd_x = 1.0 / std::sqrt(ssx / static_cast<double>(d) + eps);
            const double rstd_k = 1.0 / std::sqrt(ssk / static_cast<double>(d) + eps);
            for (int64_t i = 0; i < d; ++i) {
                xh[i] = xs[i] * rstd_x;
                kh[i] = ks[i] * rstd_k;
            }
            double dot = 0.0;
            for (int64_t i = 0; i < d; ++i) dot += xh[i] * ws[i] * kh[i];
            const double sq = sgn(dot) * std::sqrt(std::fmax(std::fabs(dot), clamp));
            const double gate = on ? sigmoid(sq) : 0.0;
            double* o = out + (n * S + s) * d;
            for (int64_t i = 0; i < d; ++i) o[i] = on ? xs[i] + gate * v[i] : xs[i];
            double* sv = saved + (n * S + s) * 4;
            sv[0] = gate;
            sv[1] = dot;
            sv[2] = rstd_x;
            sv[3] = rstd_k;
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Saved-state gate, backward  ([cuDNN-EG] layout paragraph; [TK-tests] bwd)
//
// Takes the forward's saved (gate, dot, rstd_X, rstd_key) as the values of
// those quantities, as the API does, and applies the chain rule through
//   out = X + gate*v, gate = sigmoid(sq), sq = signed sqrt with clamp,
//   dot = sum_i xh_i w_i kh_i, xh = x*rstd_X, kh = k*rstd_key.
// The saved gate is the factor that multiplied v (it enters grad_v and
// dgate = sum g*v); the gate's own derivative sigmoid'(sq) =
// sigmoid(sq)*sigmoid(-sq) is evaluated at sq recomputed from the saved dot,
// because a saved fp32 gate near 1 keeps too few bits of 1 - gate (and is
// exactly 1 once |sq| > ~17).  A zero saved gate is a masked token: its gate
// path carries no gradient (out = X there).
// The clamp's derivative is 1 where |dot| >= clamp and 0 below (a tie passes
// through, as a clamp_min does under autograd).  The RMS-norm backward is the
// generic one: dx = rstd*(dxh - xh*mean(dxh*xh)), exact also for eps > 0.
// grad_v is the sum over streams of gate_s*grad_out_s, accumulated before any
// rounding.  grad_w is summed over tokens in ascending token order.
// ---------------------------------------------------------------------------
int oracle_gate_bwd(const double* x, const double* kv, const double* w,
                    const double* saved, const double* grad_out, int64_t N,
                    int64_t S, int64_t d, double clamp, double* grad_x,
                    double* grad_kv, double* grad_w) {
    if (N < 0 || S < 1 || d < 1) return 1;
    const int64_t kvw = (S + 1) * d;
    std::vector<double> ddot_all(static_cast<size_t>(N * S));
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        std::vector<double> xh(d), kh(d), dxh(d), dkh(d);
        const double* v = kv + n * kvw + S * d;
        double* gv = grad_kv + n * kvw + S * d;
        for (int64_t i = 0; i < d; ++i) gv[i] = 0.0;
        for (int64_t s = 0; s < S; ++s) {
            const double* xs = x + (n * S + s) * d;
            const double* ks = kv + n * kvw + s * d;
            const double* ws = w + s * d;
            const double* g = grad_out + (n * S + s) * d;
            const double* sv = saved + (n * S + s) * 4;
            const double gate = sv[0], dot = sv[1], rstd_x = sv[2], rstd_k = sv[3];
            // out = X + gate * v
            double dgate = 0.0;
            for (int64_t i = 0; i < d; ++i) dgate += g[i] * v[i];
            for (int64_t i = 0; i < d; ++i) gv[i] += gate * g[i];
            // gate = sigmoid(sq), sq = sign(dot) * sqrt(max(|dot|, clamp))
            const double ad = std::fabs(dot);
            const double sq = sgn(dot) * std::sqrt(std::fmax(ad, clamp));
            const double dsq = (gate == 0.0) ? 0.0 : dgate * sigmoid(sq) * sigmoid(-sq);
            const double ddot = (ad >= clamp) ? dsq * 0.5 / std::sqrt(ad) : 0.0;
            ddot_all[static_cast<size_t>(n * S + s)] = ddot;
            // dot = sum xh * w * kh
            for (int64_t i = 0; i < d; ++i) {
                xh[i] = xs[i] * rstd_x;
                kh[i] = ks[i] * rstd_k;
                dxh[i] = ddot * ws[i] * kh[i];
                dkh[i] = ddot * ws[i] * xh[i];
            }
            // RMS-norm backward for X and for the key
            double sx = 0.0, sk = 0.0;
            for (int64_t i = 0; i < d; ++i) {
                sx += dxh[i] * xh[i];
                sk += dkh[i] * kh[i];
            }
            const double mx = sx / static_cast<double>(d);
            const double mk = sk / static_cast<double>(d);
            double* gx = grad_x + (n * S + s) * d;
            double* gk = grad_kv + n * kvw + s * d;
            for (int64_t i = 0; i < d; ++i) {
                gx[i] = g[i] + rstd_x * (dxh[i] - xh[i] * mx);
                gk[i] = rstd_k * (dkh[i] - kh[i] * mk);
            }
        }
    }
    // grad_w[s, i] = sum_n ddot[n, s] * xh[n, s, i] * kh[n, s, i], in token order
#pragma omp parallel for schedule(static)
    for (int64_t si = 0; si < S * d; ++si) {
        const int64_t s = si / d, i = si % d;
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double* sv = saved + (n * S + s) * 4;
            const double xh = x[(n * S + s) * d + i] * sv[2];
            const double kh = kv[n * kvw + s * d + i] * sv[3];
            acc += ddot_all[static_cast<size_t>(n * S + s)] * xh * kh;
        }
        grad_w[si] = acc;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// GateConv, forward  ([TileOPs] GateConv section, EngramGateConvFwdOp)
//
//   H, k, v (M, T, d); wh, wv (d); cw (4, d)
//   rrms_h = 1/sqrt(mean(H^2)+eps), rrms_k likewise; one shared weight wh
//   normalises both H and k ("RMSNorm weight for H and k").
//   alpha  = sigmoid( sum_i (H rrms_h wh)_i (k rrms_k wh)_i / sqrt(d) )
//   vhat   = alpha * v                                   (the gated value)
//   rrms_v = 1/sqrt(mean(vhat^2)+eps); u = vhat * rrms_v * wv (conv input)
//   c_t    = sum_{j=0..3} cw[j] * u_{t-3+j}, zero before the row start
//   Y      = SiLU(c) + vhat
// Readings: the gate is a plain sigmoid of the normalised dot product scaled
// by 1/sqrt(d) (no signed square root: the page names only RMSNorm gating);
// the conv has dilation 1 and no bias; tap 3 multiplies the current token.
// Outputs are exact fp64; Y and vhat are rounded to bf16 by the caller.
// ---------------------------------------------------------------------------
// Fused weight of the gate: the product of the two bf16 normalisation weights
// of the query and key sides (cuDNN Frontend "Engram saved-state gate",
// semantics paragraph: the fused weight is their FP32 product; tile-kernels
// engram fused-weight test).  weight[i] = wh[i] * we[i].
int oracle_fused_weight(const double* wh, const double* we, int64_t n, double* weight) {
    if (n < 0) return 1;
    for (int64_t i = 0; i < n; ++i) weight[i] = wh[i] * we[i];
    return 0;
}

// Gradients of the two weights from per-block grad_weight partials (tile-kernels
// engram backward test): grad_w = sum over blocks, then the product rule
// grad_wh = grad_w * we, grad_we = grad_w * wh.
int oracle_fused_weight_bwd(const double* partial, int64_t nblocks, const double* wh,
                            const double* we, int64_t n, double* grad_w, double* grad_wh,
                            double* grad_we) {
    if (n < 0 || nblocks < 0) return 1;
    for (int64_t i = 0; i < n; ++i) {
        double g = 0.0;
        for (int64_t b = 0; b < nblocks; ++b) g += partial[b * n + i];
        grad_w[i] = g;
        grad_wh[i] = g * we[i];
        grad_we[i] = g * wh[i];
    }
    return 0;
}

int oracle_gateconv_fwd(const double* H, const double* k, const double* v,
                        const double* wh, const double* wv, const double* cw,
                        int64_t M, int64_t T, int64_t d, double eps, double* Y,
                        double* vhat, double* alpha, double* rrms_h,
                        double* rrms_k, double* rrms_v) {
    if (M < 0 || T < 0 || d < 1) return 1;
    const int64_t NT = M * T;
    std::vector<double> u(static_cast<size_t>(NT * d));
    const double sqrt_d = std::sqrt(static_cast<double>(d));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < NT; ++r) {
        const double* h = H + r * d;
        const double* kk = k + r * d;
        const double* vv = v + r * d;
        double sh = 0.0, sk = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            sh += h[i] * h[i];
            sk += kk[i] * kk[i];
        }
        const double rh = 1.0 / std::sqrt(sh / static_cast<double>(d) + eps);
        const double rk = 1.0 / std::sqrt(sk / static_cast<double>(d) + eps);
        double z = 0.0;
        for (int64_t i = 0; i < d; ++i) z += (h[i] * rh * wh[i]) * (kk[i] * rk * wh[i]);
        z /= sqrt_d;
        const double a = sigmoid(z);
        double* vh = vhat + r * d;
        double sv = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            vh[i] = a * vv[i];
            sv += vh[i] * vh[i];
        }
        const double rv = 1.0 / std::sqrt(sv / static_cast<double>(d) + eps);
        double* ur = u.data() + r * d;
        for (int64_t i = 0; i < d; ++i) ur[i] = vh[i] * rv * wv[i];
        alpha[r] = a;
        rrms_h[r] = rh;
        rrms_k[r] = rk;
        rrms_v[r] = rv;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < NT; ++r) {
        const int64_t t = r % T;
        double* y = Y + r * d;
        const double* vh = vhat + r * d;
        for (int64_t i = 0; i < d; ++i) {
            double c = 0.0;
            for (int64_t j = 0; j < 4; ++j) {
                const int64_t tt = t - 3 + j;
                if (tt < 0) continue;
                c += cw[j * d + i] * u[static_cast<size_t>((r - t + tt) * d + i)];
            }
            y[i] = c * sigmoid(c) + vh[i];
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// GateConv, backward  ([TileOPs] GateConv section, EngramGateConvBwdOp)
//
// Chain rule through the forward above, evaluated at the saved activations:
// vhat, alpha, rrms_h, rrms_k, rrms_v are taken as given (vhat as the caller
// stored it); z is recomputed from H, k and the saved rrms.  Weight gradients
// are summed over all M*T tokens in ascending order.
// ---------------------------------------------------------------------------
int oracle_gateconv_bwd(const double* dY, const double* H, const double* k,
                        const double* v, const double* wh, const double* wv,
                        const double* cw, const double* vhat,
                        const double* alpha, const double* rrms_h,
                        const double* rrms_k, const double* rrms_v, int64_t M,
                        int64_t T, int64_t d, double* dH, double* dk,
                        double* dv, double* dwh, double* dwv, double* dcw) {
    if (M < 0 || T < 0 || d < 1) return 1;
    const int64_t NT = M * T;
    const double sqrt_d = std::sqrt(static_cast<double>(d));
    std::vector<double> u(static_cast<size_t>(NT * d)), dc(static_cast<size_t>(NT * d));
    // u = vhat * rrms_v * wv ;  c = causal conv of u ;  dc = dY * SiLU'(c)
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < NT; ++r)
        for (int64_t i = 0; i < d; ++i)
            u[static_cast<size_t>(r * d + i)] = vhat[r * d + i] * rrms_v[r] * wv[i];
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < NT; ++r) {
        const int64_t t = r % T;
        for (int64_t i = 0; i < d; ++i) {
            double c = 0.0;
            for (int64_t j = 0; j < 4; ++j) {
                const int64_t tt = t - 3 + j;
                if (tt < 0) continue;
                c += cw[j * d + i] * u[static_cast<size_t>((r - t + tt) * d + i)];
            }
            const double sc = sigmoid(c);
            dc[static_cast<size_t>(r * d + i)] = dY[r * d + i] * sc * (1.0 + c * (1.0 - sc));
        }
    }
    // per-token part; weight-gradient contributions are kept per token and
    // summed in token order afterwards
    std::vector<double> cwh(static_cast<size_t>(NT * d)), cwv(static_cast<size_t>(NT * d));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < NT; ++r) {
        const int64_t t = r % T;
        std::vector<double> du(d), uh(d), duh(d), dvh(d), ht(d), kt(d), dht(d), dkt(d);
        const double rv = rrms_v[r], a = alpha[r], rh = rrms_h[r], rk = rrms_k[r];
        // du_t = sum_j cw[j] * dc_{t+3-j}  (transpose of the causal conv)
        for (int64_t i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < 4; ++j) {
                const int64_t tt = t + 3 - j;
                if (tt >= T) continue;
                acc += cw[j * d + i] * dc[static_cast<size_t>((r - t + tt) * d + i)];
            }
            du[i] = acc;
        }
        // u = uh * wv with uh = vhat * rrms_v  (RMSNorm of vhat)
        double s_uh = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            uh[i] = vhat[r * d + i] * rv;
            duh[i] = du[i] * wv[i];
            cwv[static_cast<size_t>(r * d + i)] = du[i] * uh[i];
            s_uh += duh[i] * uh[i];
        }
        const double m_uh = s_uh / static_cast<double>(d);
        // Y = SiLU(c) + vhat : vhat receives dY directly plus the norm path
        double dalpha = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            dvh[i] = dY[r * d + i] + rv * (duh[i] - uh[i] * m_uh);
            dv[r * d + i] = a * dvh[i];            // vhat = alpha * v
            dalpha += dvh[i] * v[r * d + i];
        }
        const double dz = dalpha * a * (1.0 - a);
        // z = sum (ht*wh) (kt*wh) / sqrt(d), ht = H*rrms_h, kt = k*rrms_k
        double sh = 0.0, sk = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            ht[i] = H[r * d + i] * rh;
            kt[i] = k[r * d + i] * rk;
        }
        for (int64_t i = 0; i < d; ++i) {
            const double dhat_h = dz * (kt[i] * wh[i]) / sqrt_d;  // d/d(ht*wh)
            const double dhat_k = dz * (ht[i] * wh[i]) / sqrt_d;  // d/d(kt*wh)
            dht[i] = dhat_h * wh[i];
            dkt[i] = dhat_k * wh[i];
            cwh[static_cast<size_t>(r * d + i)] = dhat_h * ht[i] + dhat_k * kt[i];
            sh += dht[i] * ht[i];
            sk += dkt[i] * kt[i];
        }
        const double mh = sh / static_cast<double>(d), mk = sk / static_cast<double>(d);
        for (int64_t i = 0; i < d; ++i) {
            dH[r * d + i] = rh * (dht[i] - ht[i] * mh);
            dk[r * d + i] = rk * (dkt[i] - kt[i] * mk);
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < d; ++i) {
        double awh = 0.0, awv = 0.0;
        double ac[4] = {0.0, 0.0, 0.0, 0.0};
        for (int64_t r = 0; r < NT; ++r) {
            const int64_t t = r % T;
            awh += cwh[static_cast<size_t>(r * d + i)];
            awv += cwv[static_cast<size_t>(r * d + i)];
            // c_t = sum_j cw[j] u_{t-3+j}  ->  dcw[j] += dc_t * u_{t-3+j}
            for (int64_t j = 0; j < 4; ++j) {
                const int64_t tt = t - 3 + j;
                if (tt < 0) continue;
                ac[j] += dc[static_cast<size_t>(r * d + i)] *
                         u[static_cast<size_t>((r - t + tt) * d + i)];
            }
        }
        dwh[i] = awh;
        dwv[i] = awv;
        for (int64_t j = 0; j < 4; ++j) dcw[j * d + i] = ac[j];
    }
    return 0;
}

// GateConv decode, one token (TileOPs "Engram Operators", Decode section,
// EngramDecodeFwdOp: GEMV projection + gating + dilated conv + SiLU with a
// conv_state cache).  The page gives the interface only; this follows the
// readings of the GateConv forward above:
//   k = e W_K, v = e W_V                       (d_mem -> d, no bias)
//   alpha = sigmoid(sum (h rrms_h w_h)(k rrms_k w_h) / sqrt(d)),  vhat = alpha v
//   u = vhat rrms_v w_v,  rrms_v = 1/sqrt(mean(vhat^2) + eps)
//   c = sum_{j<w} conv_w[j] u_{t - (w-1-j) dil}   (u_t this token's u; older u
//       from conv_state, oldest first, most recent last; 0 beyond its L rows)
//   y = SiLU(c) + vhat
//   new_state = the last max_len rows of [0 (max_len - L rows), conv_state, u_t]
// e (B,d_mem), h (B,d), state (B,L,d), W_K, W_V (d_mem,d), w_h, w_v (d),
// conv_w (w,d); outputs y (B,d) and new_state (B,max_len,d) exact (the caller
// rounds; the stored u_t of a real cache is its bf16 rounding).
int oracle_decode_fwd(const double* e, const double* h, const double* state, int64_t L,
                      const double* WK, const double* WV, const double* wh, const double* wv,
                      const double* cw, int64_t B, int64_t dmem, int64_t d, int64_t max_len,
                      int64_t w, int64_t dil, double eps, double* y, double* new_state) {
    if (B < 0 || dmem < 1 || d < 1 || L < 0 || max_len < 1 || L > max_len || w < 1 || dil < 1) return 1;
    const double sqrt_d = std::sqrt(static_cast<double>(d));
    std::vector<double> k(static_cast<size_t>(d)), v(static_cast<size_t>(d)), u(static_cast<size_t>(d));
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t i = 0; i < d; ++i) {
            double sk = 0.0, sv = 0.0;
            for (int64_t m = 0; m < dmem; ++m) {
                sk += e[b * dmem + m] * WK[m * d + i];
                sv += e[b * dmem + m] * WV[m * d + i];
            }
            k[static_cast<size_t>(i)] = sk;
            v[static_cast<size_t>(i)] = sv;
        }
        double mh = 0.0, mk = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            mh += h[b * d + i] * h[b * d + i];
            mk += k[static_cast<size_t>(i)] * k[static_cast<size_t>(i)];
        }
        const double rh = 1.0 / std::sqrt(mh / static_cast<double>(d) + eps);
        const double rk = 1.0 / std::sqrt(mk / static_cast<double>(d) + eps);
        double z = 0.0;
        for (int64_t i = 0; i < d; ++i)
            z += (h[b * d + i] * rh * wh[i]) * (k[static_cast<size_t>(i)] * rk * wh[i]);
        z /= sqrt_d;
        const double alpha = sigmoid(z);
        double mv = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            const double vh = alpha * v[static_cast<size_t>(i)];
            mv += vh * vh;
        }
        const double rv = 1.0 / std::sqrt(mv / static_cast<double>(d) + eps);
        for (int64_t i = 0; i < d; ++i) {
            const double vh = alpha * v[static_cast<size_t>(i)];
            u[static_cast<size_t>(i)] = vh * rv * wv[i];
            double c = 0.0;
            for (int64_t j = 0; j < w; ++j) {
                const int64_t lag = (w - 1 - j) * dil;   // 0: this token
                double uj = 0.0;
                if (lag == 0)
                    uj = u[static_cast<size_t>(i)];
                else if (lag <= L)
                    uj = state[(b * L + (L - lag)) * d + i];
                c += cw[j * d + i] * uj;
            }
            y[b * d + i] = c * sigmoid(c) + vh;
        }
        // shift by one token: row r of the new state is row r + 1 of the old
        // state left-padded to max_len rows; the last row is u_t
        for (int64_t r = 0; r < max_len; ++r) {
            const int64_t src = r + 1 - (max_len - L);   // row of the old state
            for (int64_t i = 0; i < d; ++i) {
                double val = 0.0;
                if (r == max_len - 1)
                    val = u[static_cast<size_t>(i)];
                else if (src >= 0 && src < L)
                    val = state[(b * L + src) * d + i];
                new_state[(b * max_len + r) * d + i] = val;
            }
        }
    }
    return 0;
}

}  // extern "C"
