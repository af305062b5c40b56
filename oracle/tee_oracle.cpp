// CPU oracle of the token early-exit step: plain, slow, single-threaded C++17
// in float64. TEST INFRASTRUCTURE, NOT PRODUCT: only the tests, the smoke
// check and the benchmark's CPU-baseline / reference arms load it (through
// oracle/_native.py). It shares no code, header, table or constant with the
// CUDA library, and includes nothing but the C++ standard library.
//
// Every function is the definition written out as loops, in the order the
// source pages state it: no BLAS, no threads, no SIMD intrinsics, no blocking
// or reordering of sums (each sum runs over its index in increasing order).
// Inputs arrive as float64 (values stored in bf16 / fp16 / fp32 widen to
// float64 exactly); outputs stay unrounded, except the exit decision, which
// the TIDE notes (core module 4: the kernels accumulate in fp32) fix to fp32.
//
// Sources (page -- section):
//   River-LLM (paper.rainbus.top/paper/2604.18396): background "state
//     transition similarity"; core method; method steps 1 and 3; background
//     "PTQ" (W4A16 weights).
//   TIDE notes (dihengye.cn/.../tide): system architecture; core modules 3
//     and 4 ("Fused LayerNorm + Route", "Batch Compact", "Exit Scatter",
//     "Exit Projection"); key formulas 3 and 4; Figure 2.
//   RidgeFill (kongchang.com/.../ridgefill...): idea source; closed-form
//     ridge regression note; measured results ("identity fill").
//
// Conventions: matrices are row-major; a "row vector times matrix" product
// x W with W[k][n] is the plain sum over k. Every entry point is extern "C"
// with plain pointers and sizes; nullable pointers are marked.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

using vec = std::vector<double>;

vec zeros(int64_t n) { return vec(static_cast<size_t>(n), 0.0); }

double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

// y[m][n] = sum_k a[m][k] * b[k][n], each sum over k in increasing order.
// The k loop is outermost so that one row of b serves every row of a while it
// is in cache; every y[i][j] still adds its terms in the order k = 0, 1, ...
void matmul(const double* a, const double* b, double* y, int64_t m, int64_t k, int64_t n) {
    for (int64_t i = 0; i < m * n; ++i) y[i] = 0.0;
    for (int64_t t = 0; t < k; ++t) {
        const double* bt = b + t * n;
        for (int64_t i = 0; i < m; ++i) {
            const double ait = a[i * k + t];
            double* yi = y + i * n;
            for (int64_t j = 0; j < n; ++j) yi[j] += ait * bt[j];
        }
    }
}

// One row: x / sqrt(mean(x^2) + eps) * gamma (gamma nullable = 1).
void rms_norm_row(const double* x, const double* gamma, int64_t d, double eps, double* y) {
    double ss = 0.0;
    for (int64_t i = 0; i < d; ++i) ss += x[i] * x[i];
    const double r = 1.0 / std::sqrt(ss / double(d) + eps);
    for (int64_t i = 0; i < d; ++i) y[i] = x[i] * r * (gamma ? gamma[i] : 1.0);
}

// Rotate-half RoPE of one head of width hd at position pos: element i pairs
// with i + hd/2 and turns by pos * base^(-2i/hd) (positions from 0, no
// frequency scaling, float64 angles).
void rope_row(const double* k, int64_t hd, double pos, double base, double* y) {
    const int64_t half = hd / 2;
    for (int64_t i = 0; i < half; ++i) {
        const double inv_freq = std::pow(base, -2.0 * double(i) / double(hd));
        const double ang = pos * inv_freq;
        const double c = std::cos(ang), s = std::sin(ang);
        const double x1 = k[i], x2 = k[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- exit gates

// River-LLM, background "state transition similarity" and method step 3:
// s = <h_prev, h_cur> / (|h_prev| |h_cur|) per token (row). A zero row has no
// direction: s = 0 (it never exits).
void oc_cosine_similarity(int64_t n, int64_t d, const double* h_prev, const double* h_cur, double* s) {
    for (int64_t t = 0; t < n; ++t) {
        const double* a = h_prev + t * d;
        const double* b = h_cur + t * d;
        double dot = 0.0, na = 0.0, nb = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            dot += a[i] * b[i];
            na += a[i] * a[i];
            nb += b[i] * b[i];
        }
        const double den = std::sqrt(na) * std::sqrt(nb);
        s[t] = den > 0.0 ? dot / den : 0.0;
    }
}

// Strict score > threshold, decided on the fp32-rounded score against the
// fp32 threshold (River-LLM core method "exceeds tau"; TIDE formula 4
// "phi_k > theta"; TIDE module 4 accumulates in fp32). flag = 1 iff every
// token exits, i.e. iff min_b s_b > tau. rule 0 = per token (mask = each
// token's decision), rule 1 = batch (every mask entry = flag; River-LLM
// method step 3's min over the batch, TIDE module 3's "all tokens").
int oc_decide(int64_t n, const double* score, double threshold, int rule, uint8_t* mask, int32_t* flag) {
    if (rule != 0 && rule != 1) return 1;
    const float thr = float(threshold);
    int32_t all = n > 0 ? 1 : 0;
    for (int64_t t = 0; t < n; ++t) {
        mask[t] = float(score[t]) > thr ? 1 : 0;
        if (!mask[t]) all = 0;
    }
    if (rule == 1)
        for (int64_t t = 0; t < n; ++t) mask[t] = uint8_t(all);
    *flag = all;
    return 0;
}

// TIDE formula 3 and module 4 ("Fused LayerNorm + Route"), per token:
//   r = 1 / sqrt(mean(h^2) + eps)
//   u[c] = sum_i W_down[c][i] * (h[i] * r * gamma[i]) + b_down[c]   (c < b)
//   z = sum_c W_up[c] * SiLU(u[c]) + b_up,   SiLU(x) = x * sigmoid(x)
//   p = sigmoid(z)
// W_down is [b][d] (formula 3's W_down in R^{b x d}), W_up [b]. gamma,
// b_down, b_up nullable (the system-architecture count of d*128 + 128
// parameters per checkpoint leaves no room for them: gamma = 1, biases 0).
void oc_router_probability(int64_t n, int64_t d, int64_t b, const double* h, const double* w_down,
                           const double* w_up, const double* gamma, const double* b_down, const double* b_up,
                           double eps, double* p) {
    // u[c] = sum_i W_down[c][i] hn[i] with W_down read through its transpose, so
    // that the c loop is innermost; each u[c] still adds its terms in the order
    // i = 0, 1, ...
    vec wt = zeros(d * b);
    for (int64_t c = 0; c < b; ++c)
        for (int64_t i = 0; i < d; ++i) wt[size_t(i * b + c)] = w_down[c * d + i];
    vec hn = zeros(d);
    vec u = zeros(b);
    for (int64_t t = 0; t < n; ++t) {
        rms_norm_row(h + t * d, gamma, d, eps, hn.data());
        for (int64_t c = 0; c < b; ++c) u[size_t(c)] = 0.0;
        for (int64_t i = 0; i < d; ++i) {
            const double x = hn[size_t(i)];
            const double* wi = wt.data() + i * b;
            for (int64_t c = 0; c < b; ++c) u[size_t(c)] += wi[c] * x;
        }
        double z = 0.0;
        for (int64_t c = 0; c < b; ++c) {
            double uc = u[size_t(c)];
            if (b_down) uc += b_down[c];
            z += w_up[c] * (uc * sigmoid(uc));
        }
        if (b_up) z += b_up[0];
        p[t] = sigmoid(z);
    }
}

// TIDE formula 4, earliest-checkpoint rule: probs[c][t] is phi at checkpoint
// layer ks[c] (0-based; ks increasing; H[k+1] is layer k's output). Token t
// exits at the first checkpoint k >= k_min whose probability exceeds theta
// (fp32 decision) and has then run k + 1 layers; otherwise all n_layers.
void oc_earliest_exit(int64_t n_ck, const int64_t* ks, int64_t n, const double* probs, double theta,
                      int64_t n_layers, int64_t k_min, int64_t* depth) {
    const float thr = float(theta);
    for (int64_t t = 0; t < n; ++t) {
        depth[t] = n_layers;
        for (int64_t c = 0; c < n_ck; ++c) {
            if (ks[c] < k_min) continue;
            if (float(probs[c * n + t]) > thr) {
                depth[t] = ks[c] + 1;
                break;
            }
        }
    }
}

// TIDE Figure 2 accounting: one layer op per token per executed layer.
int64_t oc_layer_ops(int64_t n, const int64_t* depth) {
    int64_t s = 0;
    for (int64_t t = 0; t < n; ++t) s += depth[t];
    return s;
}

// ----------------------------------------------------- compaction and scatter

// TIDE module 4 "Batch Compact": rows in order, a row with mask != 0 goes to
// the exit list, the rest to the continue list (a stable split). pos_in
// (nullable = identity) carries each row's original slot into cont_pos /
// exit_pos. counts = {n_cont, n_exit}.
void oc_stable_partition(int64_t n, const uint8_t* mask, const int64_t* pos_in, int64_t* cont_rows,
                         int64_t* exit_rows, int64_t* cont_pos, int64_t* exit_pos, int64_t* counts) {
    int64_t nc = 0, ne = 0;
    for (int64_t r = 0; r < n; ++r) {
        const int64_t p = pos_in ? pos_in[r] : r;
        if (mask[r] != 0) {
            exit_rows[ne] = r;
            exit_pos[ne] = p;
            ++ne;
        } else {
            cont_rows[nc] = r;
            cont_pos[nc] = p;
            ++nc;
        }
    }
    counts[0] = nc;
    counts[1] = ne;
}

// The compacted buffer: out row i = h row rows[i].
void oc_gather_rows(int64_t m, int64_t d, const double* h, const int64_t* rows, double* out) {
    for (int64_t i = 0; i < m; ++i) std::memcpy(out + i * d, h + rows[i] * d, size_t(d) * sizeof(double));
}

// TIDE module 4 "Exit Scatter": out[exit_pos[i]] = h_src[exit_rows[i]] for
// i < n_exit; with gamma (nullable) the row first goes through the final
// RMSNorm ("Exit Projection"). Other rows of out keep their values.
void oc_exit_scatter(int64_t n_exit, int64_t d, const double* h_src, const int64_t* exit_rows,
                     const int64_t* exit_pos, const double* gamma, double eps, double* out) {
    for (int64_t i = 0; i < n_exit; ++i) {
        const double* src = h_src + exit_rows[i] * d;
        double* dst = out + exit_pos[i] * d;
        if (gamma)
            rms_norm_row(src, gamma, d, eps, dst);
        else
            std::memcpy(dst, src, size_t(d) * sizeof(double));
    }
}

// ------------------------------------------------------------------- KV fill

// W4A16 dequantisation (River-LLM background "PTQ"; the format is the reading
// taken for HQQ, which the pages name without defining): unsigned 4-bit codes,
// two per byte along the input dimension with even k in the low nibble;
// per group of `group` input rows an fp16 scale s and fp16 zero z;
// W[k][j] = (q[k][j] - z[k/group][j]) * s[k/group][j]. packed is [k/2][n].
void oc_dequant_int4(int64_t k, int64_t n, int64_t group, const uint8_t* packed, const double* scale,
                     const double* zero, double* w) {
    for (int64_t r = 0; r < k; ++r) {
        for (int64_t j = 0; j < n; ++j) {
            const uint8_t byte = packed[(r / 2) * n + j];
            const int q = (r % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
            const int64_t g = r / group;
            w[r * n + j] = (double(q) - zero[g * n + j]) * scale[g * n + j];
        }
    }
}

// RMSNorm of each of `rows` rows of width d (gamma nullable = 1).
void oc_rms_norm(int64_t rows, int64_t d, const double* x, const double* gamma, double eps, double* y) {
    for (int64_t r = 0; r < rows; ++r) rms_norm_row(x + r * d, gamma, d, eps, y + r * d);
}

// Rotate-half RoPE of `rows` heads of width hd, head r at position pos[r].
void oc_rope_rotate_half(int64_t rows, int64_t hd, const double* k, const double* pos, double base, double* y) {
    for (int64_t r = 0; r < rows; ++r) rope_row(k + r * hd, hd, pos[r], base, y + r * hd);
}

// K and V that one filled layer writes for t split-layer rows (RidgeFill idea
// source: the map predicts the layer's input, the layer's own projections
// write the cache; River-LLM method step 1: the backbone's addressing):
//   x = h W_map            (W_map [d][d]; nullable = identity, State
//                           Propagation / "identity fill")
//   x^ = RMSNorm(x) * gamma
//   k = x^ Wk (+ k_bias),  v = x^ Wv (+ v_bias)       (Wk, Wv [d][n_kv*hd])
//   each head of k: with k_norm, RMS-normalised over hd (same eps) and scaled
//   by k_norm; then RoPE at the row's position.
// k_out, v_out are [t][n_kv][hd]. k_bias, v_bias, k_norm nullable (the
// QKV-bias and QK-norm model families of RidgeFill's measured results).
void oc_fill_rows(int64_t t, int64_t d, int64_t n_kv, int64_t hd, const double* h, const double* w_map,
                  const double* gamma, const double* wk, const double* wv, const double* k_bias,
                  const double* v_bias, const double* k_norm, const double* pos, double rope_base, double eps,
                  double* k_out, double* v_out) {
    const int64_t kvw = n_kv * hd;
    vec x = zeros(t * d);
    vec xn = zeros(t * d);
    vec k = zeros(t * kvw);
    vec head = zeros(hd);
    if (w_map)
        matmul(h, w_map, x.data(), t, d, d);
    else
        for (int64_t i = 0; i < t * d; ++i) x[size_t(i)] = h[i];
    oc_rms_norm(t, d, x.data(), gamma, eps, xn.data());
    matmul(xn.data(), wk, k.data(), t, d, kvw);
    matmul(xn.data(), wv, v_out, t, d, kvw);
    for (int64_t r = 0; r < t; ++r) {
        if (k_bias)
            for (int64_t j = 0; j < kvw; ++j) k[size_t(r * kvw + j)] += k_bias[j];
        if (v_bias)
            for (int64_t j = 0; j < kvw; ++j) v_out[r * kvw + j] += v_bias[j];
        for (int64_t g = 0; g < n_kv; ++g) {
            const double* kh = k.data() + r * kvw + g * hd;
            if (k_norm) {
                rms_norm_row(kh, k_norm, hd, eps, head.data());
                kh = head.data();
            }
            rope_row(kh, hd, pos[r], rope_base, k_out + r * kvw + g * hd);
        }
    }
}

// ----------------------------------------------------------------- ridge fit

// RidgeFill, closed-form ridge regression note: W = (X^T X + lambda I)^-1 X^T Y
// for X [n][d] (split-layer states) and Y [n][dout] (a later layer's true
// inputs). A = X^T X + lambda I is factorised A = L L^T (Cholesky, lower),
// then L Z = X^T Y and L^T W = Z are solved by substitution. Returns 0, or 1
// when a pivot is not positive (A not positive definite; W is then unset).
int oc_ridge_fit(int64_t n, int64_t d, int64_t dout, const double* X, const double* Y, double lambda, double* W) {
    vec A = zeros(d * d);
    vec B = zeros(d * dout);
    vec L = zeros(d * d);
    // A[i][j] = sum_r X[r][i] X[r][j], B[i][j] = sum_r X[r][i] Y[r][j]: the row loop
    // is outermost (one row of X and Y in cache at a time), every entry still adds
    // its terms in the order r = 0, 1, ...; lambda is added after the sum.
    for (int64_t r = 0; r < n; ++r) {
        const double* xr = X + r * d;
        const double* yr = Y + r * dout;
        for (int64_t i = 0; i < d; ++i) {
            const double xi = xr[i];
            double* ai = A.data() + i * d;
            double* bi = B.data() + i * dout;
            for (int64_t j = 0; j < d; ++j) ai[j] += xi * xr[j];
            for (int64_t j = 0; j < dout; ++j) bi[j] += xi * yr[j];
        }
    }
    for (int64_t i = 0; i < d; ++i) A[size_t(i * d + i)] += lambda;
    for (int64_t j = 0; j < d; ++j) {
        double s = A[size_t(j * d + j)];
        for (int64_t k = 0; k < j; ++k) s -= L[size_t(j * d + k)] * L[size_t(j * d + k)];
        if (!(s > 0.0)) return 1;
        const double ljj = std::sqrt(s);
        L[size_t(j * d + j)] = ljj;
        for (int64_t i = j + 1; i < d; ++i) {
            double v = A[size_t(i * d + j)];
            for (int64_t k = 0; k < j; ++k) v -= L[size_t(i * d + k)] * L[size_t(j * d + k)];
            L[size_t(i * d + j)] = v / ljj;
        }
    }
    // The substitutions run on whole rows of the right-hand sides (every column
    // c at once); each entry subtracts its terms in increasing k.
    vec Z = zeros(d * dout);
    vec v = zeros(dout);
    for (int64_t i = 0; i < d; ++i) {   // L Z = B, forward
        for (int64_t c = 0; c < dout; ++c) v[size_t(c)] = B[size_t(i * dout + c)];
        for (int64_t k = 0; k < i; ++k) {
            const double lik = L[size_t(i * d + k)];
            const double* zk = Z.data() + k * dout;
            for (int64_t c = 0; c < dout; ++c) v[size_t(c)] -= lik * zk[c];
        }
        for (int64_t c = 0; c < dout; ++c) Z[size_t(i * dout + c)] = v[size_t(c)] / L[size_t(i * d + i)];
    }
    for (int64_t i = d - 1; i >= 0; --i) {   // L^T W = Z, backward
        for (int64_t c = 0; c < dout; ++c) v[size_t(c)] = Z[size_t(i * dout + c)];
        for (int64_t k = i + 1; k < d; ++k) {
            const double lki = L[size_t(k * d + i)];
            const double* wk = W + k * dout;
            for (int64_t c = 0; c < dout; ++c) v[size_t(c)] -= lki * wk[c];
        }
        for (int64_t c = 0; c < dout; ++c) W[i * dout + c] = v[size_t(c)] / L[size_t(i * d + i)];
    }
    return 0;
}

// ------------------------------------------------------------ the Exit River

// SiLU(a) = a * sigmoid(a) = a / (1 + e^-a), elementwise.
void oc_silu(int64_t n, const double* a, double* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = a[i] / (1.0 + std::exp(-a[i]));
}

// Causal decode attention of each item over its own sequence's cache layer.
// q [n][n_q][hd]; k_layer, v_layer [n_seq][n_kv][P][hd]; item i reads
// positions 0..pos[i] of sequence seq[i]; query head h reads kv head
// h / (n_q / n_kv). o[i][h] = softmax(q . K^T / sqrt(hd)) V (the softmax with
// its maximum subtracted, which leaves it unchanged).
void oc_attention(int64_t n, int64_t n_q, int64_t hd, const double* q, const double* k_layer,
                  const double* v_layer, int64_t n_kv, int64_t P, const int64_t* pos, const int64_t* seq,
                  double* o) {
    const int64_t rep = n_q / n_kv;
    vec z;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t p = pos[i], s = seq[i];
        z.assign(size_t(p + 1), 0.0);
        for (int64_t h = 0; h < n_q; ++h) {
            const int64_t g = h / rep;
            const double* qh = q + (i * n_q + h) * hd;
            const double* K = k_layer + ((s * n_kv + g) * P) * hd;
            const double* V = v_layer + ((s * n_kv + g) * P) * hd;
            double zmax = -INFINITY;
            for (int64_t m = 0; m <= p; ++m) {
                double dot = 0.0;
                for (int64_t e = 0; e < hd; ++e) dot += K[m * hd + e] * qh[e];
                z[size_t(m)] = dot / std::sqrt(double(hd));
                if (z[size_t(m)] > zmax) zmax = z[size_t(m)];
            }
            double sum = 0.0;
            for (int64_t m = 0; m <= p; ++m) {
                z[size_t(m)] = std::exp(z[size_t(m)] - zmax);
                sum += z[size_t(m)];
            }
            double* oh = o + (i * n_q + h) * hd;
            for (int64_t e = 0; e < hd; ++e) oh[e] = 0.0;
            for (int64_t m = 0; m <= p; ++m) {
                const double w = z[size_t(m)] / sum;
                for (int64_t e = 0; e < hd; ++e) oh[e] += w * V[m * hd + e];
            }
        }
    }
}

// One Exit River layer (River-LLM core method, method step 1; the block is
// read as the Llama pre-norm block of the decoder the pages measure on):
//   x = RMSNorm(h) * attn_norm;  q, k, v = x Wq, x Wk, x Wv
//   RoPE (rotate-half) on every head of q and k at the item's position
//   cache[seq][kv head][pos] <- k, v   (every item of the call before any
//                                       attention)
//   o = attention over positions 0..pos of the item's sequence
//   h1 = h + o Wo;  x2 = RMSNorm(h1) * ffn_norm
//   h' = h1 + (SiLU(x2 Wg) * (x2 Wu)) Wd
// Weights are dense float64 [in][out] (int4 weights are dequantised first by
// oc_dequant_int4); k_cache, v_cache are this layer's [n_seq][n_kv][P][hd],
// written in place. h, h_out [n][d].
void oc_exit_layer(int64_t n, int64_t d, int64_t n_q, int64_t n_kv, int64_t hd, int64_t d_ff, const double* h,
                   const double* attn_norm, const double* ffn_norm, const double* wq, const double* wk,
                   const double* wv, const double* wo, const double* wg, const double* wu, const double* wd,
                   const int64_t* pos, const int64_t* seq, int64_t P, double* k_cache, double* v_cache,
                   double rope_base, double eps, double* h_out) {
    const int64_t qw = n_q * hd, kvw = n_kv * hd;
    vec x = zeros(n * d);
    vec q = zeros(n * qw);
    vec k = zeros(n * kvw);
    vec v = zeros(n * kvw);
    vec qr = zeros(n * qw);
    vec o = zeros(n * qw);
    vec ao = zeros(n * d);
    vec h1 = zeros(n * d);
    vec x2 = zeros(n * d);
    vec gt = zeros(n * d_ff);
    vec up = zeros(n * d_ff);
    vec a = zeros(n * d_ff);
    vec down = zeros(n * d);
    oc_rms_norm(n, d, h, attn_norm, eps, x.data());
    matmul(x.data(), wq, q.data(), n, d, qw);
    matmul(x.data(), wk, k.data(), n, d, kvw);
    matmul(x.data(), wv, v.data(), n, d, kvw);
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t hh = 0; hh < n_q; ++hh)
            rope_row(q.data() + i * qw + hh * hd, hd, double(pos[i]), rope_base, qr.data() + i * qw + hh * hd);
        for (int64_t g = 0; g < n_kv; ++g) {
            double* kslot = k_cache + ((seq[i] * n_kv + g) * P + pos[i]) * hd;
            double* vslot = v_cache + ((seq[i] * n_kv + g) * P + pos[i]) * hd;
            rope_row(k.data() + i * kvw + g * hd, hd, double(pos[i]), rope_base, kslot);
            for (int64_t e = 0; e < hd; ++e) vslot[e] = v[size_t(i * kvw + g * hd + e)];
        }
    }
    oc_attention(n, n_q, hd, qr.data(), k_cache, v_cache, n_kv, P, pos, seq, o.data());
    matmul(o.data(), wo, ao.data(), n, qw, d);
    for (int64_t i = 0; i < n * d; ++i) h1[size_t(i)] = h[i] + ao[size_t(i)];
    oc_rms_norm(n, d, h1.data(), ffn_norm, eps, x2.data());
    matmul(x2.data(), wg, gt.data(), n, d, d_ff);
    matmul(x2.data(), wu, up.data(), n, d, d_ff);
    oc_silu(n * d_ff, gt.data(), a.data());
    for (int64_t i = 0; i < n * d_ff; ++i) a[size_t(i)] *= up[size_t(i)];
    matmul(a.data(), wd, down.data(), n, d_ff, d);
    for (int64_t i = 0; i < n * d; ++i) h_out[i] = h1[size_t(i)] + down[size_t(i)];
}

// Build identification (checked by the loader).
int oc_abi_version(void) { return 1; }

}  // extern "C"
