/*
 * CPU ORACLE of the fused speculative-decode verify step — test
 * infrastructure only.
 *
 * Plain, slow, fp64 C++17. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark call it; the product path never does. It
 * shares no source with the CUDA library: its own structs, its own Q4/q8
 * codecs, its own binary16 conversion, its own page allocator.
 *
 * What it computes (one verify cycle of the hybrid decoder the
 * "Fusing the whole speculative-decoding cycle into one CUDA kernel" page
 * describes, section "What shipped": main model over T = 1 + n_draft rows,
 * lm_head, greedy verification on device, commit of the recurrent state only
 * through the accepted token):
 *
 *   for every row of every sequence, in position order, in fp64:
 *     x = dequant(embedding row of the token)
 *     per layer: u = RMSNorm(x)
 *       Gated DeltaNet layer: [qkv, z, a, b] = W u; causal conv (width 4) + SiLU
 *         on qkv; q, k L2-normalised per head; alpha = sigmoid(a),
 *         beta = sigmoid(b); S <- alpha S + beta (v - alpha S k) k^T; o = S q;
 *         o' = RMSNorm_head(o) * w  (.) SiLU(z); x += W_o o'
 *       gated attention layer: q, gate, k, v = W u; RoPE on q, k; k, v stored
 *         into the paged pool as fp16 or q8; softmax(q k^T / sqrt(dh)) v over
 *         positions <= p, read back as stored; o' = attn (.) sigmoid(gate);
 *         x += W_o o'
 *       FFN: x += W_down (SiLU(W_gate u) (.) W_up u)
 *     logits = W_lm RMSNorm(x)
 *   greedy verification: g_j = argmax(row j), accepted a = longest prefix with
 *     draft_i == g_{i-1}; emitted d_1..d_a, g_a; count = a + 1.
 *   (sampling verification, for temperature > 0, is orc_sample_verify at the
 *   end of this file: it works on a sequence's logits and given uniforms.)
 *   commit: L += kept rows; recurrent state <- snapshot after the last kept row;
 *     pages wholly beyond L are freed; new pages are the lowest free ids, in row
 *     order.
 *   drafts for the next cycle (models with a multi-token-prediction block; the
 *     page's "MTP catch-up rows for accepted tokens, then n_draft MTP draft
 *     steps", restricted to the first draft_vocab tokens as its section "What
 *     shipped" states): for each accepted row i = 0..a, whose next token is g_i,
 *       m = W_fc [RMSNorm(h_i) w_h ; RMSNorm(emb(g_i)) w_e]    (h_i: the row's
 *           final hidden state before the final norm)
 *       m = one gated-attention decoder layer on m at position p_i, with its own
 *           KV layer (index n_fa in the pool)
 *       draft logits = W_lm[0:draft_vocab] RMSNorm_final'(m)
 *     draft 1 = argmax of row a's draft logits; then for j = 1 .. n_draft-1 one
 *     more pass with (previous pass's m, draft j) at position p_a + j gives
 *     draft j+1.
 *
 * Every matrix-vector product sums over k in index order; threads split only
 * the output rows. Parity pins: tests/test_oracle_pins.py.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <set>
#include <thread>
#include <vector>

extern "C" {

struct OrcLayout {
    int32_t n_layers, hidden, ffn, vocab;
    int32_t kind[64]; /* 0 Gated DeltaNet, 1 gated full attention */
    int32_t hq, hkv, dh;
    double rope_base;
    int32_t hk, hv, dk, dv, conv_w;
    int32_t tied, has_mtp, draft_vocab, n_draft;
    int32_t kv_q8, page_tokens, n_pages, max_seqs, max_pages_per_seq;
    double eps;
};

struct OrcLayerW {
    const float* attn_norm;
    const uint8_t *w_qkv, *w_z, *w_a, *w_b;
    const float* conv_w;
    const float* o_norm;
    const uint8_t *w_q, *w_g, *w_k, *w_v;
    const uint8_t* w_o;
    const float* ffn_norm;
    const uint8_t *w_gate, *w_up, *w_down;
};

struct OrcWeights {
    const uint8_t* embed;
    const float* final_norm;
    const uint8_t* lm_head; /* NULL when tied to the embedding */
    OrcLayerW layer[64];
    OrcLayerW mtp;
    const uint8_t* mtp_fc;
    const float *mtp_norm_h, *mtp_norm_e, *mtp_final_norm;
};

/* KV pool as stored; owned by the caller, the oracle writes new positions. */
struct OrcPool {
    uint16_t *k, *v;   /* fp16 [n_kv_layers][n_pages][hkv][page_tokens][dh] */
    int8_t *kq, *vq;   /* q8 codes, same shape */
    uint16_t *ks, *vs; /* q8 scales [n_kv_layers][n_pages][hkv][page_tokens][dh/32] */
};

} /* extern "C" */

namespace {

/* ------------------------------------------------------------ binary16 */

double half_value(uint16_t h) {
    const int exponent = (h >> 10) & 31;
    const int mantissa = h & 1023;
    double mag;
    if (exponent == 0)
        mag = std::ldexp(static_cast<double>(mantissa), -24);
    else if (exponent == 31)
        mag = mantissa ? NAN : INFINITY;
    else
        mag = std::ldexp(1024.0 + mantissa, exponent - 25);
    return (h & 0x8000) ? -mag : mag;
}

/* Round a double to the nearest binary16 (ties to even). */
uint16_t half_round(double x) {
    if (std::isnan(x)) return 0x7e00;
    const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
    const double a = std::fabs(x);
    /* Largest finite is 65504; its rounding boundary to infinity is 65520. */
    if (a >= 65520.0) return sign | 0x7c00;
    /* Scale so that one unit in the last place of the target is 1. */
    int e2 = a > 0 ? std::ilogb(a) : -30; /* a in [2^e2, 2^(e2+1)) */
    if (e2 < -14) e2 = -14;               /* subnormals share the 2^-24 ulp */
    const double ulp = std::ldexp(1.0, e2 - 10);
    double units = std::nearbyint(a / ulp); /* integer count of ulps */
    if (e2 == -14 && units < 1024) return sign | static_cast<uint16_t>(units);
    if (units >= 2048) { units /= 2; e2 += 1; }
    if (e2 > 15) return sign | 0x7c00;
    return sign | static_cast<uint16_t>(((e2 + 15) << 10) | (static_cast<int>(units) - 1024));
}

/* ------------------------------------------------------------ Q4 codec */

constexpr int kQ4Bytes = 144;

/* Dequantise one 256-weight super-block: w = d*sc_j*q - dmin*m_j. */
void q4_decode(const uint8_t* blk, double* w) {
    const double d = half_value(static_cast<uint16_t>(blk[0] | (blk[1] << 8)));
    const double dmin = half_value(static_cast<uint16_t>(blk[2] | (blk[3] << 8)));
    const uint8_t* field = blk + 4;
    auto bits6 = [&](int at) {
        int v = 0;
        for (int b = 0; b < 6; ++b) v |= ((field[(at + b) / 8] >> ((at + b) % 8)) & 1) << b;
        return v;
    };
    for (int j = 0; j < 8; ++j) {
        const int sc = bits6(6 * j);
        const int m = bits6(48 + 6 * j);
        const uint8_t* codes = blk + 16 + 16 * j;
        for (int i = 0; i < 32; ++i) {
            const int q = i < 16 ? (codes[i] & 15) : (codes[i - 16] >> 4);
            w[32 * j + i] = d * sc * q - dmin * m;
        }
    }
}

/* Q4 quantiser (for the generator cross-check), restated from the format:
 * per sub-block range [min(0, min w), max w] split into 15 steps; super-block
 * d, dmin are the largest step / offset over 63, in binary16; 6-bit sub-block
 * scales and mins; 4-bit codes; rounding half to even throughout. */
void q4_encode(const double* w, uint8_t* blk) {
    double step[8], offset[8];
    for (int j = 0; j < 8; ++j) {
        double lo = 0.0, hi = -INFINITY;
        for (int i = 0; i < 32; ++i) {
            lo = std::min(lo, w[32 * j + i]);
            hi = std::max(hi, w[32 * j + i]);
        }
        step[j] = (hi - lo) / 15.0;
        offset[j] = -lo;
    }
    const double max_step = *std::max_element(step, step + 8);
    const double max_off = *std::max_element(offset, offset + 8);
    const uint16_t dbits = half_round(max_step / 63.0), mbits = half_round(max_off / 63.0);
    const double d = half_value(dbits), dmin = half_value(mbits);
    int sc[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0 ? static_cast<int>(std::clamp(std::nearbyint(step[j] / d), 0.0, 63.0)) : 0;
        mn[j] = dmin > 0 ? static_cast<int>(std::clamp(std::nearbyint(offset[j] / dmin), 0.0, 63.0)) : 0;
    }
    std::memset(blk, 0, kQ4Bytes);
    blk[0] = dbits & 255; blk[1] = dbits >> 8;
    blk[2] = mbits & 255; blk[3] = mbits >> 8;
    auto put6 = [&](int at, int v) {
        for (int b = 0; b < 6; ++b)
            if ((v >> b) & 1) blk[4 + (at + b) / 8] |= static_cast<uint8_t>(1 << ((at + b) % 8));
    };
    for (int j = 0; j < 8; ++j) { put6(6 * j, sc[j]); put6(48 + 6 * j, mn[j]); }
    for (int j = 0; j < 8; ++j) {
        const double denom = d * sc[j];
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (denom > 0)
                q = static_cast<int>(std::clamp(std::nearbyint((w[32 * j + i] + dmin * mn[j]) / denom), 0.0, 15.0));
            uint8_t& byte = blk[16 + 16 * j + (i % 16)];
            byte |= static_cast<uint8_t>(i < 16 ? q : q << 4);
        }
    }
}

/* ------------------------------------------------------------ q8 codec */

/* Block of 32: d16 = f16(amax/127); q = clamp(rne(x/d16), -127, 127), 0 if
 * d16 == 0; value = d16 * q. */
void q8_encode(const double* x, int8_t* q, uint16_t* d16) {
    double amax = 0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(x[i]));
    *d16 = half_round(amax / 127.0);
    const double d = half_value(*d16);
    for (int i = 0; i < 32; ++i)
        q[i] = d == 0 ? 0 : static_cast<int8_t>(std::clamp(std::nearbyint(x[i] / d), -127.0, 127.0));
}

/* ------------------------------------------------------------ threads */

void parallel_rows(int n, int nthreads, const std::function<void(int, int)>& fn) {
    if (nthreads <= 1 || n < 64) { fn(0, n); return; }
    nthreads = std::min(nthreads, n / 16 + 1);
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) {
        const int b = static_cast<int>(static_cast<int64_t>(n) * t / nthreads);
        const int e = static_cast<int>(static_cast<int64_t>(n) * (t + 1) / nthreads);
        pool.emplace_back(fn, b, e);
    }
    for (auto& th : pool) th.join();
}

/* y[n] = sum_k W[n][k] u[k] for a Q4 matrix (rows x K), k in index order. */
void q4_matvec(const uint8_t* W, int rows, int K, const double* u, double* y, int nthreads) {
    const int nsb = K / 256;
    parallel_rows(rows, nthreads, [&](int b, int e) {
        double w[256];
        for (int n = b; n < e; ++n) {
            double acc = 0;
            for (int s = 0; s < nsb; ++s) {
                q4_decode(W + (static_cast<size_t>(n) * nsb + s) * kQ4Bytes, w);
                for (int i = 0; i < 256; ++i) acc += w[i] * u[256 * s + i];
            }
            y[n] = acc;
        }
    });
}

/* ------------------------------------------------------------ small ops */

double sigmoid(double v) { return 1.0 / (1.0 + std::exp(-v)); }
double silu(double v) { return v * sigmoid(v); }

/* y = x / sqrt(mean(x^2) + eps) * g */
void rmsnorm(const double* x, const float* g, int n, double eps, double* y) {
    double ss = 0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    const double inv = 1.0 / std::sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (g ? g[i] : 1.0);
}

/* x <- x / sqrt(sum x^2 + eps) */
void l2norm(double* x, int n, double eps) {
    double ss = 0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    const double inv = 1.0 / std::sqrt(ss + eps);
    for (int i = 0; i < n; ++i) x[i] *= inv;
}

/* Rotate-half RoPE: pairs (i, i + dh/2), angle pos * base^(-2i/dh). */
void rope(double* x, int dh, int pos, double base) {
    const int half = dh / 2;
    for (int i = 0; i < half; ++i) {
        const double theta = pos * std::pow(base, -2.0 * i / dh);
        const double c = std::cos(theta), s = std::sin(theta);
        const double a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = a * s + b * c;
    }
}

/* out = sum_j softmax_j(q . K_j / sqrt(dh)) V_j over n keys. */
void attend(const double* q, const double* K, const double* V, int n, int dh, double* out) {
    std::vector<double> score(n);
    double mx = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double s = 0;
        for (int d = 0; d < dh; ++d) s += q[d] * K[static_cast<size_t>(j) * dh + d];
        score[j] = s / std::sqrt(static_cast<double>(dh));
        mx = std::max(mx, score[j]);
    }
    double total = 0;
    for (int j = 0; j < n; ++j) { score[j] = std::exp(score[j] - mx); total += score[j]; }
    for (int d = 0; d < dh; ++d) out[d] = 0;
    for (int j = 0; j < n; ++j) {
        const double p = score[j] / total;
        for (int d = 0; d < dh; ++d) out[d] += p * V[static_cast<size_t>(j) * dh + d];
    }
}

/* One delta-rule step on a dv x dk state: S <- alpha S + beta (v - alpha S k) k^T,
 * then o = S q. */
void gdn_update(double* S, int dk, int dv, const double* q, const double* k, const double* v,
                double alpha, double beta, double* o) {
    for (int i = 0; i < dv; ++i) {
        double* row = S + static_cast<size_t>(i) * dk;
        double sk = 0;
        for (int c = 0; c < dk; ++c) sk += row[c] * k[c];
        const double delta = beta * (v[i] - alpha * sk);
        for (int c = 0; c < dk; ++c) row[c] = alpha * row[c] + delta * k[c];
        double so = 0;
        for (int c = 0; c < dk; ++c) so += row[c] * q[c];
        o[i] = so;
    }
}

/* ------------------------------------------------------------ model */

struct Seq {
    bool used = false;
    int len = 0;
    std::vector<int> pages;
    std::vector<double> S;    /* [n_gdn][hv][dv][dk] */
    std::vector<double> conv; /* [n_gdn][conv_w-1][conv_ch] */
    /* Pending verify result of the last step. */
    bool pending = false;
    int count = 0;
    std::vector<std::vector<double>> S_after, conv_after; /* per row */
    /* Drafts of the last verify step (multi-token prediction), per draft pass:
     * token, top-1 minus top-2 logit, rms of the logits, logits and the block's
     * hidden output. */
    std::vector<int> drafts;
    std::vector<double> draft_gap, draft_rms, draft_logits, draft_hidden;
};

struct Oracle {
    OrcLayout L;
    OrcWeights W;
    OrcPool P;
    int nthreads;
    int conv_ch, n_gdn, n_fa;
    std::vector<int> gdn_index, fa_index; /* layer -> index among its kind */
    std::vector<Seq> seqs;
    std::set<int> free_pages;
    std::vector<double> last_hidden; /* main-model hidden of the rows of the last step */

    size_t S_size() const { return static_cast<size_t>(n_gdn) * L.hv * L.dv * L.dk; }
    size_t conv_size() const { return static_cast<size_t>(n_gdn) * (L.conv_w - 1) * conv_ch; }
    const uint8_t* lm() const { return L.tied ? W.embed : W.lm_head; }

    void q4_row(const uint8_t* M, int K, int r, double* out) const {
        const int nsb = K / 256;
        for (int s = 0; s < nsb; ++s) q4_decode(M + (static_cast<size_t>(r) * nsb + s) * kQ4Bytes, out + 256 * s);
    }

    /* Stored element (kvl, page, head, slot, d) of K (which=0) or V (1). */
    size_t kv_index(int kvl, int page, int head, int slot, int d) const {
        return ((((static_cast<size_t>(kvl) * L.n_pages + page) * L.hkv + head) * L.page_tokens + slot) * L.dh) + d;
    }

    void kv_store(int kvl, const Seq& s, int pos, int head, const double* x, int which) {
        const int page = s.pages[pos / L.page_tokens], slot = pos % L.page_tokens;
        const size_t base = kv_index(kvl, page, head, slot, 0);
        if (L.kv_q8) {
            int8_t* q = which ? P.vq : P.kq;
            uint16_t* sc = which ? P.vs : P.ks;
            for (int b = 0; b < L.dh / 32; ++b) q8_encode(x + 32 * b, q + base + 32 * b, sc + base / 32 + b);
        } else {
            uint16_t* h = which ? P.v : P.k;
            for (int d = 0; d < L.dh; ++d) h[base + d] = half_round(x[d]);
        }
    }

    void kv_load(int kvl, const Seq& s, int pos, int head, double* x, int which) const {
        const int page = s.pages[pos / L.page_tokens], slot = pos % L.page_tokens;
        const size_t base = kv_index(kvl, page, head, slot, 0);
        if (L.kv_q8) {
            const int8_t* q = which ? P.vq : P.kq;
            const uint16_t* sc = which ? P.vs : P.ks;
            for (int d = 0; d < L.dh; ++d) x[d] = half_value(sc[(base + d) / 32]) * q[base + d];
        } else {
            const uint16_t* h = which ? P.v : P.k;
            for (int d = 0; d < L.dh; ++d) x[d] = half_value(h[base + d]);
        }
    }

    /* Gated full attention block for one row at position pos (cache layer kvl). */
    void attention_block(const OrcLayerW& lw, int kvl, Seq& s, int pos, const double* u, double* out_o) {
        const int H = L.hidden, qdim = L.hq * L.dh, kvdim = L.hkv * L.dh;
        std::vector<double> q(qdim), gate(qdim), k(kvdim), v(kvdim);
        q4_matvec(lw.w_q, qdim, H, u, q.data(), nthreads);
        q4_matvec(lw.w_g, qdim, H, u, gate.data(), nthreads);
        q4_matvec(lw.w_k, kvdim, H, u, k.data(), nthreads);
        q4_matvec(lw.w_v, kvdim, H, u, v.data(), nthreads);
        for (int h = 0; h < L.hq; ++h) rope(&q[h * L.dh], L.dh, pos, L.rope_base);
        for (int h = 0; h < L.hkv; ++h) {
            rope(&k[h * L.dh], L.dh, pos, L.rope_base);
            kv_store(kvl, s, pos, h, &k[h * L.dh], 0);
            kv_store(kvl, s, pos, h, &v[h * L.dh], 1);
        }
        const int n = pos + 1, group = L.hq / L.hkv;
        std::vector<double> K(static_cast<size_t>(n) * L.dh), V(static_cast<size_t>(n) * L.dh);
        std::vector<double> attn(qdim);
        for (int kh = 0; kh < L.hkv; ++kh) {
            for (int j = 0; j < n; ++j) {
                kv_load(kvl, s, j, kh, &K[static_cast<size_t>(j) * L.dh], 0);
                kv_load(kvl, s, j, kh, &V[static_cast<size_t>(j) * L.dh], 1);
            }
            for (int h = kh * group; h < (kh + 1) * group; ++h)
                attend(&q[h * L.dh], K.data(), V.data(), n, L.dh, &attn[h * L.dh]);
        }
        for (int i = 0; i < qdim; ++i) out_o[i] = attn[i] * sigmoid(gate[i]);
    }

    /* Feed-forward sub-layer with its residual: x += W_down (SiLU(W_gate u) (.) W_up u),
     * u = RMSNorm(x) w_ffn. */
    void feed_forward(const OrcLayerW& lw, double* x) {
        const int H = L.hidden, F = L.ffn;
        std::vector<double> u(H), y(H), g(F), up(F);
        rmsnorm(x, lw.ffn_norm, H, L.eps, u.data());
        q4_matvec(lw.w_gate, F, H, u.data(), g.data(), nthreads);
        q4_matvec(lw.w_up, F, H, u.data(), up.data(), nthreads);
        for (int i = 0; i < F; ++i) g[i] = silu(g[i]) * up[i];
        q4_matvec(lw.w_down, H, F, g.data(), y.data(), nthreads);
        for (int i = 0; i < H; ++i) x[i] += y[i];
    }

    /* One row of the main model. Updates s (KV pool, S, conv); returns logits. */
    void forward_row(Seq& s, int token, int pos, double* logits, double* hidden_out) {
        const int H = L.hidden;
        std::vector<double> x(H), u(H), y(H);
        q4_row(W.embed, H, token, x.data());
        for (int l = 0; l < L.n_layers; ++l) {
            const OrcLayerW& lw = W.layer[l];
            rmsnorm(x.data(), lw.attn_norm, H, L.eps, u.data());
            if (L.kind[l] == 0) {
                const int gi = gdn_index[l];
                const int qk = L.hk * L.dk, vd = L.hv * L.dv, cw = L.conv_w;
                std::vector<double> pre(conv_ch), c(conv_ch), z(vd), a(L.hv), b(L.hv);
                q4_matvec(lw.w_qkv, conv_ch, H, u.data(), pre.data(), nthreads);
                q4_matvec(lw.w_z, vd, H, u.data(), z.data(), nthreads);
                q4_matvec(lw.w_a, L.hv, H, u.data(), a.data(), nthreads);
                q4_matvec(lw.w_b, L.hv, H, u.data(), b.data(), nthreads);
                /* causal depthwise conv over [history..., current], then SiLU */
                double* hist = &s.conv[static_cast<size_t>(gi) * (cw - 1) * conv_ch];
                for (int ch = 0; ch < conv_ch; ++ch) {
                    double acc = 0;
                    for (int t = 0; t < cw - 1; ++t) acc += lw.conv_w[ch * cw + t] * hist[t * conv_ch + ch];
                    acc += lw.conv_w[ch * cw + cw - 1] * pre[ch];
                    c[ch] = silu(acc);
                    for (int t = 0; t + 1 < cw - 1; ++t) hist[t * conv_ch + ch] = hist[(t + 1) * conv_ch + ch];
                    hist[(cw - 2) * conv_ch + ch] = pre[ch];
                }
                for (int g = 0; g < L.hk; ++g) {
                    l2norm(&c[g * L.dk], L.dk, L.eps);
                    l2norm(&c[qk + g * L.dk], L.dk, L.eps);
                }
                std::vector<double> o(vd), on(vd);
                const int per = L.hv / L.hk;
                for (int h = 0; h < L.hv; ++h) {
                    const int g = h / per;
                    double* S = &s.S[(static_cast<size_t>(gi) * L.hv + h) * L.dv * L.dk];
                    gdn_update(S, L.dk, L.dv, &c[g * L.dk], &c[qk + g * L.dk], &c[2 * qk + h * L.dv],
                               sigmoid(a[h]), sigmoid(b[h]), &o[h * L.dv]);
                    rmsnorm(&o[h * L.dv], lw.o_norm, L.dv, L.eps, &on[h * L.dv]);
                    for (int i = 0; i < L.dv; ++i) on[h * L.dv + i] *= silu(z[h * L.dv + i]);
                }
                q4_matvec(lw.w_o, H, vd, on.data(), y.data(), nthreads);
            } else {
                std::vector<double> o(L.hq * L.dh);
                attention_block(lw, fa_index[l], s, pos, u.data(), o.data());
                q4_matvec(lw.w_o, H, L.hq * L.dh, o.data(), y.data(), nthreads);
            }
            for (int i = 0; i < H; ++i) x[i] += y[i];
            feed_forward(lw, x.data());
        }
        if (hidden_out) std::copy(x.begin(), x.end(), hidden_out);
        rmsnorm(x.data(), W.final_norm, H, L.eps, u.data());
        q4_matvec(lm(), L.vocab, H, u.data(), logits, nthreads);
    }

    /* One row of the multi-token-prediction block: h is a final hidden state
     * (before the final norm), next the token that follows it. Writes the
     * block's KV at pos into the draft KV layer; returns the block's hidden
     * output and the logits over the first draft_vocab tokens. */
    void mtp_row(Seq& s, const double* h, int next, int pos, double* h_out, double* logits) {
        const int H = L.hidden;
        std::vector<double> cat(2 * static_cast<size_t>(H)), e(H), x(H), u(H), o(L.hq * L.dh), y(H);
        rmsnorm(h, W.mtp_norm_h, H, L.eps, cat.data());
        q4_row(W.embed, H, next, e.data());
        rmsnorm(e.data(), W.mtp_norm_e, H, L.eps, cat.data() + H);
        q4_matvec(W.mtp_fc, H, 2 * H, cat.data(), x.data(), nthreads);
        rmsnorm(x.data(), W.mtp.attn_norm, H, L.eps, u.data());
        attention_block(W.mtp, n_fa, s, pos, u.data(), o.data());
        q4_matvec(W.mtp.w_o, H, L.hq * L.dh, o.data(), y.data(), nthreads);
        for (int i = 0; i < H; ++i) x[i] += y[i];
        feed_forward(W.mtp, x.data());
        std::copy(x.begin(), x.end(), h_out);
        rmsnorm(x.data(), W.mtp_final_norm, H, L.eps, u.data());
        q4_matvec(lm(), L.draft_vocab, H, u.data(), logits, nthreads);
    }

    /* Drafts for the next cycle of a verified sequence: catch-up rows 0..a of
     * this step (row i: hidden h_i, next token g_i, position p_i), then
     * n_draft - 1 one-row passes chained on the block's own hidden output. */
    void mtp_drafts(Seq& s, int a, const double* hidden, const int* g, const int* pos);

    void commit(Seq& s, int keep) {
        s.len += keep;
        s.S = s.S_after[keep - 1];
        s.conv = s.conv_after[keep - 1];
        s.pending = false;
        s.S_after.clear();
        s.conv_after.clear();
        release_pages(s);
    }

    /* Pages wholly at or beyond the sequence length go back to the pool. */
    void release_pages(Seq& s) {
        const int need = (s.len + L.page_tokens - 1) / L.page_tokens;
        while (static_cast<int>(s.pages.size()) > need) {
            free_pages.insert(s.pages.back());
            s.pages.pop_back();
        }
    }
};

int argmax_lowest(const double* v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

void Oracle::mtp_drafts(Seq& s, int a, const double* hidden, const int* g, const int* pos) {
    const int H = L.hidden, DV = L.draft_vocab, n = L.n_draft;
    std::vector<double> lg(DV), hin(H), hout(H);
    s.drafts.assign(n, 0);
    s.draft_gap.assign(n, 0.0);
    s.draft_rms.assign(n, 0.0);
    s.draft_logits.assign(static_cast<size_t>(n) * DV, 0.0);
    s.draft_hidden.assign(static_cast<size_t>(n) * H, 0.0);
    int token = -1;
    for (int j = 0; j < n; ++j) {
        if (j == 0) {
            for (int i = 0; i <= a; ++i)
                mtp_row(s, hidden + static_cast<size_t>(i) * H, g[i], pos[i], hout.data(), lg.data());
        } else {
            mtp_row(s, hin.data(), token, pos[a] + j, hout.data(), lg.data());
        }
        token = argmax_lowest(lg.data(), DV);
        double second = -INFINITY, ss = 0;
        for (int v = 0; v < DV; ++v) {
            ss += lg[v] * lg[v];
            if (v != token) second = std::max(second, lg[v]);
        }
        s.drafts[j] = token;
        s.draft_gap[j] = lg[token] - second;
        s.draft_rms[j] = std::sqrt(ss / DV);
        std::copy(lg.begin(), lg.end(), s.draft_logits.begin() + static_cast<size_t>(j) * DV);
        std::copy(hout.begin(), hout.end(), s.draft_hidden.begin() + static_cast<size_t>(j) * H);
        hin = hout;
    }
}

} /* namespace */

extern "C" {

enum { ORC_OK = 0, ORC_INVALID = -1, ORC_NO_PAGES = -2 };

void* orc_create(const OrcLayout* L, const OrcWeights* W, const OrcPool* P, int nthreads) {
    if (L->has_mtp && (L->n_draft < 0 || L->draft_vocab < 1 || L->draft_vocab > L->vocab)) return nullptr;
    auto* o = new Oracle();
    o->L = *L;
    o->W = *W;
    o->P = *P;
    o->nthreads = nthreads;
    o->conv_ch = 2 * L->hk * L->dk + L->hv * L->dv;
    o->n_gdn = o->n_fa = 0;
    o->gdn_index.assign(L->n_layers, -1);
    o->fa_index.assign(L->n_layers, -1);
    for (int l = 0; l < L->n_layers; ++l) {
        if (L->kind[l] == 0) o->gdn_index[l] = o->n_gdn++;
        else o->fa_index[l] = o->n_fa++;
    }
    o->seqs.resize(L->max_seqs);
    for (int p = 0; p < L->n_pages; ++p) o->free_pages.insert(p);
    return o;
}

void orc_free(void* h) { delete static_cast<Oracle*>(h); }

/* Install a sequence: its length, page table and recurrent state (fp32 inputs). */
int orc_seq_set(void* h, int seq, int length, const int* pages, int n_pages, const float* S,
                const float* conv) {
    auto* o = static_cast<Oracle*>(h);
    if (seq < 0 || seq >= o->L.max_seqs) return ORC_INVALID;
    Seq& s = o->seqs[seq];
    for (int p : s.pages) o->free_pages.insert(p);
    s = Seq();
    s.used = true;
    s.len = length;
    for (int i = 0; i < n_pages; ++i) {
        if (!o->free_pages.count(pages[i])) return ORC_INVALID;
        o->free_pages.erase(pages[i]);
        s.pages.push_back(pages[i]);
    }
    s.S.assign(o->S_size(), 0.0);
    s.conv.assign(o->conv_size(), 0.0);
    if (S)
        for (size_t i = 0; i < o->S_size(); ++i) s.S[i] = S[i];
    if (conv)
        for (size_t i = 0; i < o->conv_size(); ++i) s.conv[i] = conv[i];
    return ORC_OK;
}

/* Copy out a sequence's committed state. Any pointer may be NULL. */
int orc_seq_get(void* h, int seq, int* length, int* pages, int* n_pages, double* S, double* conv) {
    auto* o = static_cast<Oracle*>(h);
    if (seq < 0 || seq >= o->L.max_seqs) return ORC_INVALID;
    const Seq& s = o->seqs[seq];
    if (length) *length = s.len;
    if (n_pages) *n_pages = static_cast<int>(s.pages.size());
    if (pages) std::copy(s.pages.begin(), s.pages.end(), pages);
    if (S) std::copy(s.S.begin(), s.S.end(), S);
    if (conv) std::copy(s.conv.begin(), s.conv.end(), conv);
    return ORC_OK;
}

/* Explicit commit of the kept rows (1 <= n_keep <= count) of pending sequences. */
int orc_commit(void* h, int n, const int* seq_ids, const int* n_keep) {
    auto* o = static_cast<Oracle*>(h);
    for (int i = 0; i < n; ++i) {
        if (seq_ids[i] < 0 || seq_ids[i] >= o->L.max_seqs) return ORC_INVALID;
        Seq& s = o->seqs[seq_ids[i]];
        if (!s.pending || n_keep[i] < 1 || n_keep[i] > s.count) return ORC_INVALID;
    }
    for (int i = 0; i < n; ++i) o->commit(o->seqs[seq_ids[i]], n_keep[i]);
    return ORC_OK;
}

/*
 * One verify step. Rows of a sequence must be contiguous, with consecutive
 * positions starting at its length. flags: 0 decode/verify row, 1 prompt
 * chunk row, 2 prompt chunk row that ends its prompt (emits one token).
 * Outputs (caller sized): out_tokens [n_rows] grouped per sequence in order of
 * first appearance, out_counts [number of sequences], and per row (optional):
 * logits [n_rows][vocab], hidden [n_rows][hidden], argmax, gap (top1 - top2),
 * rms (root mean square of the row's logits).
 */
int orc_step(void* h, int n_rows, const int* tokens, const int* positions, const int* seq_ids,
             const uint8_t* flags, int* out_tokens, int* out_counts, double* logits,
             double* hidden, int* argmax, double* gap, double* rms) {
    auto* o = static_cast<Oracle*>(h);
    const OrcLayout& L = o->L;
    if (n_rows <= 0) return ORC_INVALID;
    /* group rows by sequence (contiguous runs) */
    std::vector<int> order, start, count;
    for (int r = 0; r < n_rows; ++r) {
        const int sid = seq_ids[r];
        if (sid < 0 || sid >= L.max_seqs || !o->seqs[sid].used) return ORC_INVALID;
        if (tokens[r] < 0 || tokens[r] >= L.vocab) return ORC_INVALID;
        if (r == 0 || sid != seq_ids[r - 1]) {
            if (std::find(order.begin(), order.end(), sid) != order.end()) return ORC_INVALID;
            order.push_back(sid);
            start.push_back(r);
            count.push_back(0);
        }
        count.back()++;
    }
    for (size_t i = 0; i < order.size(); ++i) {
        Seq& s = o->seqs[order[i]];
        const bool prefill = flags && flags[start[i]] != 0;
        for (int j = 0; j < count[i]; ++j) {
            const int r = start[i] + j;
            if ((flags && flags[r] != 0) != prefill) return ORC_INVALID;
            if (flags && flags[r] == 2 && j != count[i] - 1) return ORC_INVALID;
        }
        if (s.pending) o->commit(s, s.count); /* auto-commit */
        for (int j = 0; j < count[i]; ++j)
            if (positions[start[i] + j] != s.len + j) return ORC_INVALID;
    }
    /* page allocation: lowest free id, in row order. With drafting, the last
     * row of a verified sequence also reserves the positions its draft passes
     * may write (up to its own position + n_draft - 1). */
    const bool drafting = L.has_mtp && L.n_draft > 0;
    for (int r = 0; r < n_rows; ++r) {
        Seq& s = o->seqs[seq_ids[r]];
        const bool last = r + 1 == n_rows || seq_ids[r + 1] != seq_ids[r];
        const bool verify = !(flags && flags[r] != 0);
        const int reach = positions[r] + (drafting && last && verify ? L.n_draft - 1 : 0);
        const int need = reach / L.page_tokens + 1;
        while (static_cast<int>(s.pages.size()) < need) {
            if (o->free_pages.empty() || static_cast<int>(s.pages.size()) >= L.max_pages_per_seq)
                return ORC_NO_PAGES;
            s.pages.push_back(*o->free_pages.begin());
            o->free_pages.erase(o->free_pages.begin());
        }
    }
    std::vector<double> lg(static_cast<size_t>(L.vocab));
    std::vector<int> g(n_rows);
    o->last_hidden.assign(static_cast<size_t>(n_rows) * L.hidden, 0.0);
    int out_at = 0;
    for (size_t i = 0; i < order.size(); ++i) {
        Seq& s = o->seqs[order[i]];
        s.S_after.clear();
        s.conv_after.clear();
        for (int j = 0; j < count[i]; ++j) {
            const int r = start[i] + j;
            o->forward_row(s, tokens[r], positions[r], lg.data(), &o->last_hidden[static_cast<size_t>(r) * L.hidden]);
            s.S_after.push_back(s.S);
            s.conv_after.push_back(s.conv);
            g[r] = argmax_lowest(lg.data(), L.vocab);
            if (logits) std::copy(lg.begin(), lg.end(), logits + static_cast<size_t>(r) * L.vocab);
            if (hidden) std::copy(o->last_hidden.begin() + static_cast<size_t>(r) * L.hidden,
                                  o->last_hidden.begin() + static_cast<size_t>(r + 1) * L.hidden,
                                  hidden + static_cast<size_t>(r) * L.hidden);
            if (argmax) argmax[r] = g[r];
            if (gap || rms) {
                double second = -INFINITY, ss = 0;
                for (int vv = 0; vv < L.vocab; ++vv) {
                    ss += lg[vv] * lg[vv];
                    if (vv != g[r]) second = std::max(second, lg[vv]);
                }
                if (gap) gap[r] = lg[g[r]] - second;
                if (rms) rms[r] = std::sqrt(ss / L.vocab);
            }
        }
        /* state was advanced through every row; the snapshots decide what is kept */
        const bool prefill = flags && flags[start[i]] != 0;
        if (prefill) {
            const int last = start[i] + count[i] - 1;
            const bool emits = flags[last] == 2;
            if (emits) out_tokens[out_at++] = g[last];
            out_counts[i] = emits ? 1 : 0;
            s.pending = true;
            s.count = count[i];
            o->commit(s, count[i]);
        } else {
            int a = 0;
            while (a + 1 < count[i] && tokens[start[i] + a + 1] == g[start[i] + a]) ++a;
            for (int j = 1; j <= a; ++j) out_tokens[out_at++] = tokens[start[i] + j];
            out_tokens[out_at++] = g[start[i] + a];
            out_counts[i] = a + 1;
            s.pending = true;
            s.count = a + 1;
            if (drafting)
                o->mtp_drafts(s, a, &o->last_hidden[static_cast<size_t>(start[i]) * L.hidden], &g[start[i]],
                              &positions[start[i]]);
        }
    }
    return ORC_OK;
}

/* Drafts computed by the last verify step of a sequence (models with a
 * multi-token-prediction block): per draft pass its token, top-1 minus top-2
 * draft logit, rms of the draft logits, the logits [n_draft][draft_vocab] and
 * the block's hidden output [n_draft][hidden]. Pointers may be NULL. */
int orc_drafts(void* h, int seq, int* drafts, double* gap, double* rms, double* logits, double* hidden) {
    auto* o = static_cast<Oracle*>(h);
    if (seq < 0 || seq >= o->L.max_seqs) return ORC_INVALID;
    const Seq& s = o->seqs[seq];
    if (s.drafts.empty()) return ORC_INVALID;
    if (drafts) std::copy(s.drafts.begin(), s.drafts.end(), drafts);
    if (gap) std::copy(s.draft_gap.begin(), s.draft_gap.end(), gap);
    if (rms) std::copy(s.draft_rms.begin(), s.draft_rms.end(), rms);
    if (logits) std::copy(s.draft_logits.begin(), s.draft_logits.end(), logits);
    if (hidden) std::copy(s.draft_hidden.begin(), s.draft_hidden.end(), hidden);
    return ORC_OK;
}

/* ------------------------------------------------- building blocks for pins */

void orc_q4_decode(const uint8_t* blocks, int64_t n_blocks, double* out) {
    for (int64_t b = 0; b < n_blocks; ++b) q4_decode(blocks + b * kQ4Bytes, out + b * 256);
}

void orc_q4_encode(const double* w, int64_t n_blocks, uint8_t* out) {
    for (int64_t b = 0; b < n_blocks; ++b) q4_encode(w + b * 256, out + b * kQ4Bytes);
}

void orc_q4_matvec(const uint8_t* W, int rows, int K, const double* u, double* y, int nthreads) {
    q4_matvec(W, rows, K, u, y, nthreads);
}

void orc_q8_encode(const double* x, int64_t n_blocks, int8_t* q, uint16_t* d16) {
    for (int64_t b = 0; b < n_blocks; ++b) q8_encode(x + 32 * b, q + 32 * b, d16 + b);
}

uint16_t orc_half_round(double x) { return half_round(x); }
double orc_half_value(uint16_t hbits) { return half_value(hbits); }

void orc_rmsnorm(const double* x, const float* g, int n, double eps, double* y) { rmsnorm(x, g, n, eps, y); }
void orc_l2norm(double* x, int n, double eps) { l2norm(x, n, eps); }
void orc_rope(double* x, int dh, int pos, double base) { rope(x, dh, pos, base); }
void orc_attend(const double* q, const double* K, const double* V, int n, int dh, double* out) {
    attend(q, K, V, n, dh, out);
}
void orc_gdn_update(double* S, int dk, int dv, const double* q, const double* k, const double* v,
                    double alpha, double beta, double* o) {
    gdn_update(S, dk, dv, q, k, v, alpha, beta, o);
}
double orc_sigmoid(double v) { return sigmoid(v); }
double orc_silu(double v) { return silu(v); }

int orc_n_free_pages(void* h) { return static_cast<int>(static_cast<Oracle*>(h)->free_pages.size()); }

/*
 * Speculative SAMPLING verification of one sequence's T rows. Page "UPDATE:
 * Qwen 3.8 27B 140 tok/s on single RTX 3090 Megakernel: KL divergence 0.0009
 * vs llama.cpp", section "Decode accuracy": with sampling the output keeps the
 * distribution of sampling without drafts; page "OpenJet's CUDA megakernel
 * runs 4 coding agents on one RTX 3090", section "Caveats": top_k capped at
 * 32. The drafts are single proposals (prompt-lookup or the MTP head's
 * greedy choice), so the rule is the standard one for a draft proposed with
 * probability 1:
 *   p_j = softmax over the top_k largest logits of row j (ties: lower token
 *         id first) of logits / temperature, zero elsewhere.
 *   for i = 0 .. T-2, d = drafts[i] (the token of row i+1, proposed with
 *   certainty): accept when u[i][0] < p_i(d); otherwise emit x drawn from
 *   the residual p_i(x) for x != d (renormalised by 1 - p_i(d)) by inverse
 *   CDF over ascending token ids with u[i][1], and stop.
 *   all accepted: emit a bonus drawn from p_{T-1} with u[T-1][1].
 * out receives the accepted drafts then the last token; returns the count
 * (accepted + 1), or -1 on a bad argument. logits fp64 [T][V], u [T][2].
 */
static void topk_probs(const double* row, int V, double temperature, int top_k, std::vector<double>& p) {
    std::vector<int> idx(V);
    for (int x = 0; x < V; ++x) idx[x] = x;
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return row[a] > row[b]; });
    p.assign(V, 0.0);
    const int k = std::min(top_k, V);
    const double m = row[idx[0]] / temperature;
    double z = 0;
    for (int j = 0; j < k; ++j) {
        p[idx[j]] = std::exp(row[idx[j]] / temperature - m);
        z += p[idx[j]];
    }
    for (int j = 0; j < k; ++j) p[idx[j]] /= z;
}

static int draw(const std::vector<double>& w, double total, double u) {
    /* the first token whose running sum of w exceeds u * total */
    double acc = 0;
    int last = -1;
    for (int x = 0; x < static_cast<int>(w.size()); ++x) {
        if (w[x] <= 0) continue;
        acc += w[x];
        last = x;
        if (u * total < acc) return x;
    }
    return last;
}

int orc_sample_verify(const double* logits, int T, int V, const int* drafts, double temperature, int top_k,
                      const double* u, int* out) {
    if (T < 1 || V < 1 || !(temperature > 0) || top_k < 1 || !logits || !u || !out || (T > 1 && !drafts))
        return -1;
    std::vector<double> p;
    for (int i = 0; i + 1 < T; ++i) {
        topk_probs(logits + static_cast<size_t>(i) * V, V, temperature, top_k, p);
        const int d = drafts[i];
        if (d < 0 || d >= V) return -1;
        if (u[2 * i] < p[d]) {
            out[i] = d;
            continue;
        }
        const double pd = p[d];
        p[d] = 0;
        out[i] = draw(p, 1.0 - pd, u[2 * i + 1]);
        return i + 1;
    }
    topk_probs(logits + static_cast<size_t>(T - 1) * V, V, temperature, top_k, p);
    out[T - 1] = draw(p, 1.0, u[2 * (T - 1) + 1]);
    return T;
}

} /* extern "C" */
