// Plain, slow CPU decoder in float32 arithmetic -- TEST INFRASTRUCTURE ONLY.
//
// Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
// --impl reference legs load this library.  It shares no source, header,
// table or constant with the CUDA path; it is built by oracle/build.py
// with g++ -O3 -ffp-contract=off (no fused multiply-add, no fast-math), so
// every float operation below is one IEEE-754 single-precision operation
// rounded to nearest even, in the order written.
//
// What it computes.  Forward(W, h) of Theorem 4.1 in "Vosti: Specifying,
// Implementing, and Verifying Deterministic LLM Inference" (深入解析 Vosti,
// §二, Theorem 4.1 engine-step preservation): the logits of a cold causal
// forward over the token history h from an empty KV cache, and fKV(W, h, p)
// (same page, §五 5.1): the per-layer K/V at position p of that forward.
// Batch invariance reaches the same mathematical result as the plain
// definition, so this is the plain definition, written for one position
// after another with no tiling, splitting or reordering:
//
//   * matrix products: for each output element, float32 products of two
//     bf16 values (exact in float32) added in ascending k into a zero
//     float32 accumulator;
//   * attention of the row at position p, query head h (kv head
//     h / (Hq / Hkv)): s_j = (q . k_j) * (1 / sqrt(hd)) for the visible keys
//     j = lo .. p (lo = 0, or max(0, p - w + 1) on a layer with a window of
//     w keys, 深入解析 Vosti §六 6.2), m = max s_j, e_j = exp(s_j - m),
//     o = (sum_j e_j v_j) / (sum_j e_j), every sum in ascending j;
//   * the model's dtype is bf16 (§二 Definition 2.1 puts the numeric dtype
//     into W), so each module output is rounded to bf16, round to nearest
//     even: norm outputs, projections, RoPE, attention, GLU, residual adds;
//     the logits stay float32.
//
// Per decoder layer (Llama block; Gemma-3 deltas in brackets):
//   a = rms(x); q,k,v = bf16(a Wqkv^T); [q,k = rms_head(q), rms_head(k)]
//   q,k = bf16(rope(q,k)); o = bf16(attention); h = bf16(o Wo^T)
//   [h = rms(h, post_attn)]; x = bf16(x + h)
//   a = rms(x); g,u = bf16(a Wgu^T); z = bf16(act(g) u); h = bf16(z Wd^T)
//   [h = rms(h, post_ffn)]; x = bf16(x + h)
//   logits = rms(x) Wlm^T (float32)
// rms(x) = bf16(x * (1 / sqrt(sum(x^2) / d + eps)) * g), g = w or (1 + w);
// RoPE rotates the pairs (i, i + hd/2) by p * theta^(-2i/hd), its cos / sin
// evaluated in double and rounded to float32.  Layer i of a model with a
// window w > 0 and a local:global period P > 0 is a local (windowed,
// theta_local) layer unless (i + 1) % P == 0; P = 6 gives the five local
// layers to one global layer of the Gemma-3-4B configuration.
//
// Threads split output features (or query heads) only, so no element's
// order of operations depends on the thread count.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ------------------------------------------------------------ bf16 format
// bfloat16 is the top half of a float32: same sign and 8-bit exponent, 7
// stored mantissa bits.
float bf16_value(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round to nearest, ties to even, from the bit pattern: add just under half
// a unit of the kept part, plus one if the kept part is odd, then truncate.
// A carry out of the mantissa moves to the next binade (or to infinity).
uint16_t bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) {                   // infinity or NaN
    return static_cast<uint16_t>((u >> 16) | ((u & 0x007fffffu) ? 0x0040u : 0u));
  }
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

float bf16(float f) { return bf16_value(bf16_bits(f)); }

// ------------------------------------------------------------ threads
template <class Fn>
void parallel_for(int64_t n, int threads, Fn fn) {
  if (threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  const int nt = static_cast<int>(std::min<int64_t>(threads, n));
  std::vector<std::thread> pool;
  for (int w = 0; w < nt; ++w)
    pool.emplace_back([=, &fn] {
      for (int64_t i = w; i < n; i += nt) fn(i);
    });
  for (auto& t : pool) t.join();
}

// ------------------------------------------------------------ modules
bool layer_is_local(int layer, int window, int period) {
  return window > 0 && period > 0 && (layer + 1) % period != 0;
}

// y[t][j] = sum over k ascending of x[t][k] * W[j][k]; W is bf16 [N][K].
void linear(const float* x, int64_t n, int K, const uint16_t* W, int N, float* y, int threads) {
  // x transposed to [k][t], so that for a fixed (j, k) the n running sums
  // (one per token, each its own chain in k) touch adjacent floats.
  std::vector<float> xt(static_cast<size_t>(K) * n);
  for (int64_t t = 0; t < n; ++t)
    for (int k = 0; k < K; ++k) xt[static_cast<size_t>(k) * n + t] = x[t * K + k];
  parallel_for(N, threads, [&](int64_t j) {
    std::vector<float> acc(n, 0.0f);
    const uint16_t* w = W + j * static_cast<int64_t>(K);
    for (int k = 0; k < K; ++k) {
      const float wk = bf16_value(w[k]);
      const float* xk = &xt[static_cast<size_t>(k) * n];
      for (int64_t t = 0; t < n; ++t) acc[t] = acc[t] + xk[t] * wk;
    }
    for (int64_t t = 0; t < n; ++t) y[t * N + j] = acc[t];
  });
}

// One row of RMSNorm over d elements with gains g (already 1 + w where the
// model uses offset gains).
void rms_row(const float* x, int d, const float* g, float eps, bool round, float* y) {
  float s = 0.0f;
  for (int i = 0; i < d; ++i) s = s + x[i] * x[i];
  const float inv = 1.0f / std::sqrt(s / static_cast<float>(d) + eps);
  for (int i = 0; i < d; ++i) {
    const float v = (x[i] * inv) * g[i];
    y[i] = round ? bf16(v) : v;
  }
}

std::vector<float> gains(const uint16_t* w, int n, bool offset) {
  std::vector<float> g(n);
  for (int i = 0; i < n; ++i) g[i] = offset ? 1.0f + bf16_value(w[i]) : bf16_value(w[i]);
  return g;
}

// x: [n][H][hd] rotated in place by position pos[t].
void rope_rows(float* x, int64_t n, int H, int hd, const int32_t* pos, double theta, bool round) {
  const int half = hd / 2;
  for (int64_t t = 0; t < n; ++t)
    for (int i = 0; i < half; ++i) {
      const double ang = static_cast<double>(pos[t]) * std::pow(theta, -2.0 * i / hd);
      const float c = static_cast<float>(std::cos(ang)), s = static_cast<float>(std::sin(ang));
      for (int h = 0; h < H; ++h) {
        float* r = x + (t * H + h) * hd;
        const float x1 = r[i], x2 = r[i + half];
        const float y1 = x1 * c - x2 * s;
        const float y2 = x2 * c + x1 * s;
        r[i] = round ? bf16(y1) : y1;
        r[i + half] = round ? bf16(y2) : y2;
      }
    }
}

// Attention of rows at positions pos[t] over a bf16 cache K/V [P][Hkv][hd]
// holding every position up to the largest pos.  out: [n][Hq][hd];
// probs (optional): [n][Hq][P], the softmax weights, 0 off the visible range.
void attention_rows(const float* q, int64_t n, int Hq, int hd, const uint16_t* K, const uint16_t* V, int64_t P,
                    int Hkv, const int32_t* pos, int window, bool round, float* out, float* probs, int threads) {
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(hd)));
  const int rep = Hq / Hkv;
  parallel_for(n * Hq, threads, [&](int64_t th) {
    const int64_t t = th / Hq;
    const int h = static_cast<int>(th % Hq), g = h / rep;
    const int64_t p = pos[t];
    const int64_t lo = window > 0 ? std::max<int64_t>(0, p - window + 1) : 0;
    const float* qr = q + th * hd;
    std::vector<float> s(p - lo + 1);
    for (int64_t j = lo; j <= p; ++j) {
      const uint16_t* kr = K + (j * Hkv + g) * hd;
      float dot = 0.0f;
      for (int i = 0; i < hd; ++i) dot = dot + qr[i] * bf16_value(kr[i]);
      s[j - lo] = dot * scale;
    }
    float m = s[0];
    for (float v : s) m = std::max(m, v);
    float l = 0.0f;
    for (float& v : s) {
      v = std::exp(v - m);
      l = l + v;
    }
    float* o = out + th * hd;
    for (int i = 0; i < hd; ++i) {
      float acc = 0.0f;
      for (int64_t j = lo; j <= p; ++j) acc = acc + s[j - lo] * bf16_value(V[(j * Hkv + g) * hd + i]);
      const float v = acc / l;
      o[i] = round ? bf16(v) : v;
    }
    if (probs) {
      float* pr = probs + th * P;
      for (int64_t j = 0; j < P; ++j) pr[j] = 0.0f;
      for (int64_t j = lo; j <= p; ++j) pr[j] = s[j - lo] / l;
    }
  });
}

float silu(float g) { return g / (1.0f + std::exp(-g)); }

// tanh form of GELU: 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
float gelu_tanh(float g) {
  const float c = static_cast<float>(std::sqrt(2.0 / 3.14159265358979323846));
  const float inner = c * (g + 0.044715f * (g * g * g));
  return (0.5f * g) * (1.0f + std::tanh(inner));
}

}  // namespace

extern "C" {

// Model configuration.  act: 0 SwiGLU (silu(g) u), 1 GeGLU (tanh GELU).
struct oc_spec {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  int32_t act, qk_norm, embed_scale, norm_offset, sandwich_norm;
  int32_t sliding_window, local_global_period;
  float rms_eps;
  double rope_theta, rope_theta_local;
};

// Weight table (bf16 bit patterns, row-major [out][in]): [0] embed [V][d],
// [1] final_norm [d], [2] lm_head [V][d]; then for layer l at 3 + 10 l:
// attn_norm, wqkv [(Hq + 2 Hkv) hd][d] (q heads, k heads, v heads), q_norm,
// k_norm, wo [d][Hq hd], post_attn_norm, ffn_norm, w_gate_up [2F][d] (gate
// rows then up rows), w_down [d][F], post_ffn_norm.  Absent tensors: null.
enum { W_EMBED = 0, W_FINAL = 1, W_LM = 2, W_LAYER0 = 3, W_PER_LAYER = 10 };
enum { L_ATTN_NORM, L_QKV, L_QNORM, L_KNORM, L_WO, L_POST_ATTN, L_FFN_NORM, L_GATE_UP, L_DOWN, L_POST_FFN };

int oc_layer_is_local(int layer, int window, int period) { return layer_is_local(layer, window, period) ? 1 : 0; }

void oc_round_bf16(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = bf16(x[i]);
}

void oc_rmsnorm(const float* x, int64_t rows, int d, const float* w, float eps, int offset, int round, float* y) {
  std::vector<float> g(d);
  for (int i = 0; i < d; ++i) g[i] = offset ? 1.0f + w[i] : w[i];
  for (int64_t r = 0; r < rows; ++r) rms_row(x + r * d, d, g.data(), eps, round != 0, y + r * d);
}

void oc_linear(const float* x, int64_t n, int K, const uint16_t* W, int N, float* y, int threads) {
  linear(x, n, K, W, N, y, threads);
}

void oc_rope(const float* x, int64_t n, int H, int hd, const int32_t* pos, double theta, int round, float* y) {
  std::memcpy(y, x, sizeof(float) * n * H * hd);
  rope_rows(y, n, H, hd, pos, theta, round != 0);
}

void oc_attention(const float* q, int64_t n, int Hq, int hd, const uint16_t* K, const uint16_t* V, int64_t P,
                  int Hkv, const int32_t* pos, int window, int round, float* out, float* probs, int threads) {
  attention_rows(q, n, Hq, hd, K, V, P, Hkv, pos, window, round != 0, out, probs, threads);
}

void oc_glu(const float* g, const float* u, int64_t n, int act, float* z) {
  for (int64_t i = 0; i < n; ++i) z[i] = bf16((act ? gelu_tanh(g[i]) : silu(g[i])) * u[i]);
}

// One step of the cold causal forward: tokens[0..n) at positions start ..
// start + n - 1, continuing from the bf16 K/V of positions [0, start) held
// in kc / vc ([n_layers][cap][Hkv][hd] each).  The step writes the K/V of
// its own positions there, and the float32 logits of the R rows listed in
// rows (indices into tokens) to logits [R][V].  Returns 0, or -1 if the
// cache cannot hold start + n positions or an argument is out of range.
int oc_step(const oc_spec* s, const uint16_t* const* w, const int32_t* tokens, int64_t n, int64_t start,
            uint16_t* kc, uint16_t* vc, int64_t cap, const int32_t* rows, int64_t R, float* logits, int threads) {
  const int d = s->d_model, Hq = s->n_heads, Hkv = s->n_kv_heads, hd = s->head_dim, F = s->ffn_dim;
  const int qkv = (Hq + 2 * Hkv) * hd;
  if (n < 1 || start < 0 || start + n > cap || Hkv <= 0 || Hq % Hkv) return -1;
  for (int64_t t = 0; t < n; ++t)
    if (tokens[t] < 0 || tokens[t] >= s->vocab) return -1;
  for (int64_t r = 0; r < R; ++r)
    if (rows[r] < 0 || rows[r] >= n) return -1;
  const bool off = s->norm_offset != 0;
  std::vector<int32_t> pos(n);
  for (int64_t t = 0; t < n; ++t) pos[t] = static_cast<int32_t>(start + t);

  std::vector<float> x(n * d), a(n * d), h(n * d);
  const float escale = bf16(static_cast<float>(std::sqrt(static_cast<double>(d))));
  for (int64_t t = 0; t < n; ++t)
    for (int i = 0; i < d; ++i) {
      const float e = bf16_value(w[W_EMBED][static_cast<int64_t>(tokens[t]) * d + i]);
      x[t * d + i] = s->embed_scale ? bf16(e * escale) : e;
    }
  auto rms = [&](const float* in, int64_t nrows, int dim, const uint16_t* wt, float* out) {
    const std::vector<float> g = gains(wt, dim, off);
    for (int64_t r = 0; r < nrows; ++r) rms_row(in + r * dim, dim, g.data(), s->rms_eps, true, out + r * dim);
  };
  auto round_all = [](std::vector<float>& v) {
    for (float& e : v) e = bf16(e);
  };

  std::vector<float> proj(n * qkv), q(n * Hq * hd), kn(n * Hkv * hd), vn(n * Hkv * hd), o(n * Hq * hd);
  std::vector<float> gu(n * 2 * F), z(n * F);
  for (int l = 0; l < s->n_layers; ++l) {
    const uint16_t* const* lw = w + W_LAYER0 + W_PER_LAYER * l;
    const bool local = layer_is_local(l, s->sliding_window, s->local_global_period);
    const int window = local ? s->sliding_window : 0;
    const double theta = local ? s->rope_theta_local : s->rope_theta;

    rms(x.data(), n, d, lw[L_ATTN_NORM], a.data());
    linear(a.data(), n, d, lw[L_QKV], qkv, proj.data(), threads);
    round_all(proj);
    for (int64_t t = 0; t < n; ++t) {
      std::memcpy(&q[t * Hq * hd], &proj[t * qkv], sizeof(float) * Hq * hd);
      std::memcpy(&kn[t * Hkv * hd], &proj[t * qkv + Hq * hd], sizeof(float) * Hkv * hd);
      std::memcpy(&vn[t * Hkv * hd], &proj[t * qkv + (Hq + Hkv) * hd], sizeof(float) * Hkv * hd);
    }
    if (s->qk_norm) {  // per head, over its hd elements
      rms(q.data(), n * Hq, hd, lw[L_QNORM], q.data());
      rms(kn.data(), n * Hkv, hd, lw[L_KNORM], kn.data());
    }
    rope_rows(q.data(), n, Hq, hd, pos.data(), theta, true);
    rope_rows(kn.data(), n, Hkv, hd, pos.data(), theta, true);
    uint16_t* Kl = kc + static_cast<int64_t>(l) * cap * Hkv * hd;
    uint16_t* Vl = vc + static_cast<int64_t>(l) * cap * Hkv * hd;
    for (int64_t t = 0; t < n; ++t)
      for (int i = 0; i < Hkv * hd; ++i) {
        Kl[(start + t) * Hkv * hd + i] = bf16_bits(kn[t * Hkv * hd + i]);
        Vl[(start + t) * Hkv * hd + i] = bf16_bits(vn[t * Hkv * hd + i]);
      }
    attention_rows(q.data(), n, Hq, hd, Kl, Vl, start + n, Hkv, pos.data(), window, true, o.data(), nullptr,
                   threads);
    linear(o.data(), n, Hq * hd, lw[L_WO], d, h.data(), threads);
    round_all(h);
    if (s->sandwich_norm) rms(h.data(), n, d, lw[L_POST_ATTN], h.data());
    for (int64_t i = 0; i < n * d; ++i) x[i] = bf16(x[i] + h[i]);

    rms(x.data(), n, d, lw[L_FFN_NORM], a.data());
    linear(a.data(), n, d, lw[L_GATE_UP], 2 * F, gu.data(), threads);
    round_all(gu);
    for (int64_t t = 0; t < n; ++t)
      for (int f = 0; f < F; ++f) {
        const float g = gu[t * 2 * F + f], u = gu[t * 2 * F + F + f];
        z[t * F + f] = bf16((s->act ? gelu_tanh(g) : silu(g)) * u);
      }
    linear(z.data(), n, F, lw[L_DOWN], d, h.data(), threads);
    round_all(h);
    if (s->sandwich_norm) rms(h.data(), n, d, lw[L_POST_FFN], h.data());
    for (int64_t i = 0; i < n * d; ++i) x[i] = bf16(x[i] + h[i]);
  }
  if (R > 0) {
    std::vector<float> xr(R * d), ar(R * d);
    for (int64_t r = 0; r < R; ++r) std::memcpy(&xr[r * d], &x[static_cast<int64_t>(rows[r]) * d], sizeof(float) * d);
    rms(xr.data(), R, d, w[W_FINAL], ar.data());
    linear(ar.data(), R, d, w[W_LM], s->vocab, logits, threads);
  }
  return 0;
}

}  // extern "C"
