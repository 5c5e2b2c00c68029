// CPU oracle of the sparse embedding layer (DLRM-style) -- TEST INFRASTRUCTURE ONLY.
//
// Plain, single-threaded, slow on purpose: std::unordered_map for IDs and keys, plain
// loops for pooling, the dot interaction and Adagrad, every sum accumulated in double.
// Only tests/, the smoke check and the CPU-baseline leg of the benchmark load this file's
// library; the CUDA library never does, and the two share no code.
//
// What it follows (page = one of the source web pages, named by title):
//  * HugeCTR interview (zhidx), section 2 "large sparse features": an embedding maps each
//    categorical ID to a numeric vector that sits before the feature interaction; IDs of
//    unknown range are first identified through a hash table.
//  * Merlin Distributed Embeddings article, "Background": embedding lookup is bound by
//    memory bandwidth; "synthetic model benchmark": global batch 65536 with Adagrad.
//  * DeepRec announcement, "EmbeddingVariable": dynamic-vocabulary hash table whose new
//    features start from the initializer value (generally 0).
//  * OneEmbedding article, "operator optimisation" and "usability": the pairwise dot
//    feature interaction takes (dense features, embeddings).
//
// Readings where the pages are silent, each stated in full here (Rn is only a label that
// tests and messages use to name the reading):
//  R1  static rows start at U(lo,hi) from a counter-based splitmix64 stream (spec below)
//  R3  Adagrad: acc += g^2, then w -= lr*g/(sqrt(acc)+eps)
//  R4  duplicate IDs in a batch: gradients summed first, one update per unique row
//  R5  bag index b*T+t, table-local IDs, pooled [B][T][D]
//  R6  mean divides by the bag length L (invalid IDs count in L, add 0); L=0 gives 0
//  R7  interaction vectors x0 = dense, x1..xT = pooled; pairs (i,j), i>j, i-major
//  R9  a new hashed key starts at w = hash_init (0) and acc = init_acc (0.1)
//  R10 hashed keys live in [0, 2^63); a negative key is rejected
//  R14 row-wise Adagrad: a += mean_j g_j^2, one fp32 accumulator per row
//  R15 bf16 storage: round to nearest even on every store
//  R17 every floating output comes with a magnitude (sum of absolute terms) for the
//      tolerance test |gpu - ref| <= tol * max(|ref|, magnitude); a stored parameter
//      element keeps the magnitude of the update that last wrote it, element by element
//  R19 feature admission (DeepRec announcement, "EmbeddingVariable": admission methods are
//      named, not defined): every hashed key counts its lookups over all backward steps;
//      a key's row takes the Adagrad update of a step only if its count, this step's
//      lookups included, has reached the admission minimum (0 or 1: always).  Until then
//      the row keeps its initial value.
//  R21 int8 row codec (Merlin Distributed Embeddings article, opening section: embedding
//      rows exchanged between GPUs in reduced precision; the exchange format is not given):
//      per row of d fp32 values, scale = max|x| / 127 and code = x / scale rounded to the
//      nearest integer (ties to even), clamped to [-127, 127]; a zero row has scale 0 and
//      codes 0; decoding gives code * scale.  Both steps are fp32 operations (IEEE
//      division and multiplication), so the codes are fixed bit for bit.
//  R23 Adagrad Decay (DeepRec announcement, "Adagrad Decay Optimizer": the accumulator is
//      discounted by period, every sample of one period with the same discount; the rule is
//      not given): backward step n (1, 2, ...) belongs to period (n - 1) / period_steps; when
//      a row is updated, its accumulator is first multiplied by rate^(periods since the
//      period of its previous update, counted from period 0 for a row never updated), then
//      the step adds g^2 (per element) or mean g^2 (row-wise) as in R3 / R14.
//  R22 cross interaction (OneFlow OneEmbedding article, "operator optimisation":
//      FusedCrossFeatureInteraction, with the cross layer of "Deep & Cross Network for Ad
//      Click Predictions"): per sample, x_next = x0 * (xl . w) + b + xl over vectors of
//      width K; the backward follows by the chain rule.
//  R20 feature eviction (same passage, "eviction strategies" named, not defined): backward
//      steps are numbered 1, 2, ...; each key records the last step that counted it.  An
//      eviction between steps removes every key whose idle time (current step - last
//      step) exceeds max_idle (when max_idle > 0) or whose count is below min_count; a key
//      looked up again later starts afresh (initial row, zero count).
//
// Precision: arithmetic in double; parameters are stored in the table's declared type
// (fp32, or bf16 by rounding the double result to float and then to bf16).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <unordered_map>
#include <vector>

namespace {

// flag bits reported by oracle calls (same meaning as the device status flags)
constexpr uint32_t F_ID_RANGE = 1u;    // static ID outside [0, rows)
constexpr uint32_t F_BAD_KEY = 2u;     // hashed key outside [0, 2^63)
constexpr uint32_t F_TABLE_FULL = 4u;  // no free slot for a new key
constexpr uint32_t F_STATE = 0x100u;   // backward without a forward

// SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
// OOPSLA 2014): state_n = seed + n * gamma, output = mix(state_n).
uint64_t splitmix_output(uint64_t seed, uint64_t n) {
  uint64_t z = seed + n * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Initial value of element `col` of row `id` in table `t` (reading R1):
//   counter c = ((t << 40) + id) * 512 + col,  z = output number c+1 of the stream,
//   u = (z >> 40) / 2^24 (exact in float),  v = lo + (hi - lo) * u  in float arithmetic,
//   one rounding per operation (the file is built with -ffp-contract=off).
float init_value(uint64_t seed, int t, int64_t id, int col, float lo, float hi) {
  uint64_t c = ((((uint64_t)t) << 40) + (uint64_t)id) * 512ull + (uint64_t)col;
  uint64_t z = splitmix_output(seed, c + 1);
  volatile float u = (float)(uint32_t)(z >> 40) * (1.0f / 16777216.0f);
  volatile float width = hi - lo;
  volatile float prod = width * u;
  volatile float v = lo + prod;
  return v;
}

// bf16 round to nearest, ties to even, by integer arithmetic on the float's bits.
uint16_t bf16_rne(float x) {
  uint32_t b;
  std::memcpy(&b, &x, 4);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

float bf16_to_float(uint16_t h) {
  uint32_t b = ((uint32_t)h) << 16;
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}

struct Model {
  int T = 0, D = 0;
  int hashed = 0, bf16 = 0, mean = 0, rowwise = 0;
  int64_t capacity = 0;
  double lr = 0, eps = 0;
  float init_acc = 0, lo = 0, hi = 0, hash_init = 0;
  uint64_t seed = 0;
  std::vector<int64_t> rows, base;  // static: rows per table, global row base
  // parameter store, lazily materialised: key -> index into the pools.
  // key = global row (base[t] + id) for static tables, the raw int64 key when hashed.
  std::unordered_map<uint64_t, int64_t> index;
  std::vector<uint64_t> keys;
  std::vector<float> w, acc;        // [n][D] and [n][D] (per element) or [n] (row-wise)
  std::vector<double> mag_w, mag_acc;  // per element, same shapes as w and acc: magnitude of
                                       // the update that last wrote the element (R17)
  std::vector<uint64_t> freq;       // per row (hashed): lookups counted so far (R19)
  std::vector<int64_t> last_step;   // per row (hashed): last backward step that counted it (R20)
  uint32_t admit_min = 0;           // R19
  double decay_rate = 1.0;          // R23 (1: no decay)
  int64_t decay_period = 0;         // R23 steps per period (0: no decay)
  std::vector<int64_t> last_period; // per row: period of its last update (R23)
  int64_t step = 0;                 // backward steps completed (R20)
  // last forward: one record per valid lookup
  std::vector<uint64_t> lk_key;
  std::vector<int64_t> lk_bag;
  std::vector<double> lk_scale;
  int64_t last_batch = -1;
  bool have_fwd = false;

  int acc_width() const { return rowwise ? 1 : D; }

  int64_t table_of_row(uint64_t row) const {
    int64_t t = (int64_t)(std::upper_bound(base.begin(), base.end(), (int64_t)row) - base.begin()) - 1;
    return t;
  }

  float stored(double v) const {
    float f = (float)v;
    return bf16 ? bf16_to_float(bf16_rne(f)) : f;
  }

  int64_t add_row(uint64_t key, int t, int64_t id) {
    int64_t n = (int64_t)keys.size();
    keys.push_back(key);
    for (int c = 0; c < D; ++c) {
      float v = hashed ? hash_init : init_value(seed, t, id, c, lo, hi);
      w.push_back(hashed ? stored(v) : (bf16 ? bf16_to_float(bf16_rne(v)) : v));
    }
    for (int c = 0; c < acc_width(); ++c) acc.push_back(init_acc);
    mag_w.insert(mag_w.end(), (size_t)D, 0.0);
    mag_acc.insert(mag_acc.end(), (size_t)acc_width(), 0.0);
    freq.push_back(0);
    last_step.push_back(0);
    last_period.push_back(0);
    index.emplace(key, n);
    return n;
  }
};

}  // namespace

extern "C" {

uint64_t orc_splitmix64(uint64_t seed, uint64_t n) { return splitmix_output(seed, n); }

float orc_init_value(uint64_t seed, int t, int64_t id, int col, float lo, float hi) {
  return init_value(seed, t, id, col, lo, hi);
}

uint16_t orc_bf16_rne(float x) { return bf16_rne(x); }

void* orc_create(int T, const int64_t* rows, int D, int hashed, int64_t capacity, int bf16,
                 int mean, int rowwise, double lr, double eps, float init_acc, float lo,
                 float hi, float hash_init, uint64_t seed) {
  Model* m = new Model();
  m->T = T;
  m->D = D;
  m->hashed = hashed;
  m->capacity = capacity;
  m->bf16 = bf16;
  m->mean = mean;
  m->rowwise = rowwise;
  m->lr = lr;
  m->eps = eps;
  m->init_acc = init_acc;
  m->lo = lo;
  m->hi = hi;
  m->hash_init = hash_init;
  m->seed = seed;
  if (!hashed) {
    m->rows.assign(rows, rows + T);
    m->base.assign(T + 1, 0);
    for (int t = 0; t < T; ++t) m->base[t + 1] = m->base[t] + rows[t];
  }
  return m;
}

void orc_destroy(void* h) { delete (Model*)h; }

int64_t orc_num_rows(void* h) { return (int64_t)((Model*)h)->keys.size(); }

// Forward: map IDs (static range check or hashed find-or-insert), gather and pool.
// ids: [nnz] bag-major; offsets: [B*T+1] or NULL (one ID per bag).
// pooled, mag: [B][T][D] doubles (mag = sum of |terms|, divided by L for mean).
// Returns the OR of the flag bits raised.
uint32_t orc_forward(void* h, const int64_t* ids, const int32_t* offsets, int64_t B,
                     double* pooled, double* mag) {
  Model* m = (Model*)h;
  const int T = m->T, D = m->D;
  uint32_t flags = 0;
  m->lk_key.clear();
  m->lk_bag.clear();
  m->lk_scale.clear();
  for (int64_t bag = 0; bag < B * T; ++bag) {
    const int t = (int)(bag % T);
    const int64_t beg = offsets ? offsets[bag] : bag;
    const int64_t end = offsets ? offsets[bag + 1] : bag + 1;
    const int64_t L = end - beg;
    std::vector<double> s(D, 0.0), a(D, 0.0);
    for (int64_t i = beg; i < end; ++i) {
      const int64_t id = ids[i];
      uint64_t key;
      int64_t r;
      if (!m->hashed) {
        if (id < 0 || id >= m->rows[t]) {
          flags |= F_ID_RANGE;
          continue;
        }
        key = (uint64_t)(m->base[t] + id);
        auto it = m->index.find(key);
        r = (it == m->index.end()) ? m->add_row(key, t, id) : it->second;
      } else {
        if (id < 0) {
          flags |= F_BAD_KEY;
          continue;
        }
        key = (uint64_t)id;
        auto it = m->index.find(key);
        if (it == m->index.end()) {
          if ((int64_t)m->index.size() >= m->capacity) {  // live keys (R20 removes some)
            flags |= F_TABLE_FULL;
            continue;
          }
          r = m->add_row(key, 0, 0);
        } else {
          r = it->second;
        }
      }
      // magnitude of a stored element: |w|, or the magnitude of the update that wrote it
      for (int c = 0; c < D; ++c) {
        const double v = m->w[(size_t)r * D + c];
        s[c] += v;
        a[c] += std::max(std::fabs(v), m->mag_w[(size_t)r * D + c]);
      }
      m->lk_key.push_back(key);
      m->lk_bag.push_back(bag);
      m->lk_scale.push_back((m->mean && L > 0) ? 1.0 / (double)L : 1.0);
    }
    for (int c = 0; c < D; ++c) {
      double v = s[c], av = a[c];
      if (m->mean && L > 0) {
        v /= (double)L;
        av /= (double)L;
      }
      if (pooled) pooled[bag * D + c] = v;
      if (mag) mag[bag * D + c] = av;
    }
  }
  m->last_batch = B;
  m->have_fwd = true;
  return flags;
}

// Magnitudes of the interaction inputs: |dense|, and for pooled vectors the larger of
// |pooled| and the pooled magnitude from orc_forward (when given).
static void load_x(const float* dense, const double* pooled, const double* pmag, int64_t b,
                   int T, int D, std::vector<double>& X, std::vector<double>& M) {
  for (int k = 0; k < D; ++k) {
    X[k] = dense[b * D + k];
    M[k] = std::fabs(X[k]);
  }
  for (int t = 0; t < T; ++t)
    for (int k = 0; k < D; ++k) {
      const double v = pooled[(b * T + t) * D + k];
      X[(size_t)(t + 1) * D + k] = v;
      M[(size_t)(t + 1) * D + k] = std::max(std::fabs(v), pmag ? pmag[(b * T + t) * D + k] : 0.0);
    }
}

// Pairwise dot interaction of one batch (reading R7).
// dense: [B][D] floats; pooled: [B][T][D] doubles; pmag: pooled magnitudes or NULL.
// out, mag: [B][D + P] doubles with P = F(F-1)/2, F = T+1.
void orc_interact(const float* dense, const double* pooled, const double* pmag, int64_t B,
                  int T, int D, double* out, double* mag) {
  const int F = T + 1;
  const int64_t P = (int64_t)F * (F - 1) / 2;
  const int64_t W = D + P;
  std::vector<double> X((size_t)F * D), M((size_t)F * D);
  for (int64_t b = 0; b < B; ++b) {
    load_x(dense, pooled, pmag, b, T, D, X, M);
    for (int k = 0; k < D; ++k) {
      out[b * W + k] = X[k];
      if (mag) mag[b * W + k] = std::fabs(X[k]);
    }
    int64_t p = 0;
    for (int i = 1; i < F; ++i) {
      for (int j = 0; j < i; ++j) {
        double s = 0.0, a = 0.0;
        for (int k = 0; k < D; ++k) {
          s += X[(size_t)i * D + k] * X[(size_t)j * D + k];
          a += M[(size_t)i * D + k] * M[(size_t)j * D + k];
        }
        out[b * W + D + p] = s;
        if (mag) mag[b * W + D + p] = a;
        ++p;
      }
    }
  }
}

// Backward of the interaction (chain rule of orc_interact):
//   G[i][j] = G[j][i] = dout[D + pair(i,j)] for i > j, G[i][i] = 0,
//   dX_i = sum_j G[i][j] x_j,  d_dense = dX_0 + dout[0:D],  d_pooled[t] = dX_{t+1}.
void orc_interact_backward(const float* dout, const float* dense, const double* pooled,
                           const double* pmag, int64_t B, int T, int D, double* d_dense,
                           double* d_pooled, double* mag_dense, double* mag_pooled) {
  const int F = T + 1;
  const int64_t P = (int64_t)F * (F - 1) / 2;
  const int64_t W = D + P;
  std::vector<double> X((size_t)F * D), M((size_t)F * D), G((size_t)F * F);
  for (int64_t b = 0; b < B; ++b) {
    load_x(dense, pooled, pmag, b, T, D, X, M);
    std::fill(G.begin(), G.end(), 0.0);
    int64_t p = 0;
    for (int i = 1; i < F; ++i)
      for (int j = 0; j < i; ++j) {
        G[(size_t)i * F + j] = dout[b * W + D + p];
        G[(size_t)j * F + i] = dout[b * W + D + p];
        ++p;
      }
    for (int i = 0; i < F; ++i) {
      for (int k = 0; k < D; ++k) {
        double s = 0.0, a = 0.0;
        for (int j = 0; j < F; ++j) {
          s += G[(size_t)i * F + j] * X[(size_t)j * D + k];
          a += std::fabs(G[(size_t)i * F + j]) * M[(size_t)j * D + k];
        }
        if (i == 0) {
          d_dense[b * D + k] = s + (double)dout[b * W + k];
          if (mag_dense) mag_dense[b * D + k] = a + std::fabs((double)dout[b * W + k]);
        } else {
          d_pooled[(b * T + (i - 1)) * D + k] = s;
          if (mag_pooled) mag_pooled[(b * T + (i - 1)) * D + k] = a;
        }
      }
    }
  }
}

// Backward + sparse Adagrad over the lookups recorded by the last orc_forward.
// d_pooled, mag: [B][T][D] doubles (mag may be NULL: magnitudes then taken as |d_pooled|).
// Gradient of a row = sum over its lookups of scale * d_pooled[bag] (reading R4), in
// lookup order; then one Adagrad step per touched row (readings R3, R14).
uint32_t orc_backward_adagrad(void* h, const double* d_pooled, const double* mag) {
  Model* m = (Model*)h;
  if (!m->have_fwd) return F_STATE;
  const int D = m->D;
  m->step += 1;
  std::map<uint64_t, std::pair<std::vector<double>, std::vector<double>>> grads;
  std::map<uint64_t, uint64_t> lookups;  // per key: lookups of this batch (R19)
  for (size_t q = 0; q < m->lk_key.size(); ++q) {
    lookups[m->lk_key[q]] += 1;
    auto& e = grads[m->lk_key[q]];
    if (e.first.empty()) {
      e.first.assign(D, 0.0);
      e.second.assign(D, 0.0);
    }
    const int64_t bag = m->lk_bag[q];
    const double sc = m->lk_scale[q];
    for (int c = 0; c < D; ++c) {
      const double g = d_pooled[bag * D + c];
      e.first[c] += sc * g;
      e.second[c] += sc * (mag ? mag[bag * D + c] : std::fabs(g));
    }
  }
  for (auto& kv : grads) {
    const int64_t r = m->index.at(kv.first);
    if (m->hashed) {  // R19, R20: count the lookups, stamp the step, gate the update
      m->freq[r] += lookups[kv.first];
      m->last_step[r] = m->step;
      if (m->admit_min > 1 && m->freq[r] < m->admit_min) continue;
    }
    const std::vector<double>& g = kv.second.first;
    const std::vector<double>& gm = kv.second.second;
    float* w = &m->w[(size_t)r * D];
    // R23: discount the accumulator by the periods since the row's last update
    double f = 1.0;
    if (m->decay_period > 0) {
      const int64_t period = (m->step - 1) / m->decay_period;
      f = std::pow(m->decay_rate, (double)(period - m->last_period[r]));
      m->last_period[r] = period;
    }
    // magnitudes (reading R17), element by element: of the old state (|value|, or the
    // magnitude of the update that wrote it) plus the absolute size of this step's terms
    double* mw = &m->mag_w[(size_t)r * D];
    if (!m->rowwise) {
      float* a = &m->acc[(size_t)r * D];
      double* ma = &m->mag_acc[(size_t)r * D];
      for (int c = 0; c < D; ++c) {
        const double acc_new = (double)a[c] * f + g[c] * g[c];
        const double denom = std::sqrt(acc_new) + m->eps;
        const double w_new = (double)w[c] - m->lr * g[c] / denom;
        mw[c] = std::max(std::fabs((double)w[c]), mw[c]) + m->lr * gm[c] / denom;
        ma[c] = std::max((double)a[c], ma[c]) * f + gm[c] * gm[c];
        a[c] = (float)acc_new;
        w[c] = m->stored(w_new);
      }
    } else {
      float* a = &m->acc[(size_t)r];
      double* ma = &m->mag_acc[(size_t)r];
      double sq = 0.0, sqm = 0.0;
      for (int c = 0; c < D; ++c) {
        sq += g[c] * g[c];
        sqm += gm[c] * gm[c];
      }
      const double acc_new = (double)a[0] * f + sq / (double)D;
      const double denom = std::sqrt(acc_new) + m->eps;
      for (int c = 0; c < D; ++c) {
        const double w_new = (double)w[c] - m->lr * g[c] / denom;
        mw[c] = std::max(std::fabs((double)w[c]), mw[c]) + m->lr * gm[c] / denom;
        w[c] = m->stored(w_new);
      }
      ma[0] = std::max((double)a[0], ma[0]) * f + sqm / (double)D;
      a[0] = (float)acc_new;
    }
  }
  m->have_fwd = false;
  return 0;
}

// R22: one cross layer.  x0, xl, out: [B][K]; w, b: [K]; out and its magnitude in double.
void orc_cross_forward(const float* x0, const float* xl, const float* w, const float* b,
                       int64_t B, int K, double* out, double* mag) {
  for (int64_t r = 0; r < B; ++r) {
    double s = 0.0, sa = 0.0;  // xl . w and its magnitude
    for (int k = 0; k < K; ++k) {
      s += (double)xl[r * K + k] * w[k];
      sa += std::fabs((double)xl[r * K + k] * w[k]);
    }
    for (int k = 0; k < K; ++k) {
      const double a = x0[r * K + k];
      out[r * K + k] = a * s + b[k] + xl[r * K + k];
      if (mag) mag[r * K + k] = std::fabs(a) * sa + std::fabs((double)b[k]) + std::fabs((double)xl[r * K + k]);
    }
  }
}

// R22 backward: with s = xl . w and t = x0 . dout per sample,
// dxl = dout + w t, dx0 = dout s, dw = sum over samples of xl t, db = sum of dout.
void orc_cross_backward(const float* x0, const float* xl, const float* w, const float* dout,
                        int64_t B, int K, double* dx0, double* dxl, double* dw, double* db,
                        double* mag_dx0, double* mag_dxl, double* mag_dw, double* mag_db) {
  for (int k = 0; k < K; ++k) dw[k] = db[k] = mag_dw[k] = mag_db[k] = 0.0;
  for (int64_t r = 0; r < B; ++r) {
    double s = 0.0, sa = 0.0, t = 0.0, ta = 0.0;
    for (int k = 0; k < K; ++k) {
      s += (double)xl[r * K + k] * w[k];
      sa += std::fabs((double)xl[r * K + k] * w[k]);
      t += (double)x0[r * K + k] * dout[r * K + k];
      ta += std::fabs((double)x0[r * K + k] * dout[r * K + k]);
    }
    for (int k = 0; k < K; ++k) {
      const double g = dout[r * K + k];
      dxl[r * K + k] = g + (double)w[k] * t;
      mag_dxl[r * K + k] = std::fabs(g) + std::fabs((double)w[k]) * ta;
      dx0[r * K + k] = g * s;
      mag_dx0[r * K + k] = std::fabs(g) * sa;
      dw[k] += (double)xl[r * K + k] * t;
      mag_dw[k] += std::fabs((double)xl[r * K + k]) * ta;
      db[k] += g;
      mag_db[k] += std::fabs(g);
    }
  }
}

// R21: int8 codes and per-row scales of n rows of d floats (row-major).
void orc_quantize_rows(const float* x, int64_t n, int d, int8_t* q, float* scale) {
  for (int64_t r = 0; r < n; ++r) {
    const float* row = x + r * d;
    float amax = 0.0f;
    for (int c = 0; c < d; ++c) amax = std::max(amax, std::fabs(row[c]));
    const float s = amax / 127.0f;
    scale[r] = s;
    for (int c = 0; c < d; ++c) {
      float v = s > 0.0f ? std::nearbyint(row[c] / s) : 0.0f;  // default rounding: ties to even
      v = std::min(127.0f, std::max(-127.0f, v));
      q[r * d + c] = (int8_t)v;
    }
  }
}

// R21: decoded rows, x = code * scale in fp32.
void orc_dequantize_rows(const int8_t* q, const float* scale, int64_t n, int d, float* x) {
  for (int64_t r = 0; r < n; ++r)
    for (int c = 0; c < d; ++c) x[r * d + c] = (float)q[r * d + c] * scale[r];
}

// R23: accumulator discount `rate` per period of `period_steps` backward steps (0: off).
void orc_set_adagrad_decay(void* h, double rate, int64_t period_steps) {
  ((Model*)h)->decay_rate = rate;
  ((Model*)h)->decay_period = period_steps;
}

// R19: admission minimum of a hashed model (0 or 1: every key is admitted at once).
void orc_set_admission(void* h, uint32_t admit_min) { ((Model*)h)->admit_min = admit_min; }

// R20: remove every hashed key idle for more than max_idle steps (max_idle > 0) or counted
// fewer than min_count times.  Returns the number of keys removed.
int64_t orc_evict(void* h, uint32_t max_idle, uint32_t min_count) {
  Model* m = (Model*)h;
  if (!m->hashed) return 0;
  std::vector<uint64_t> gone;
  for (auto& kv : m->index) {
    const int64_t r = kv.second;
    const bool idle = max_idle > 0 && m->step - m->last_step[r] > (int64_t)max_idle;
    if (idle || m->freq[r] < min_count) gone.push_back(kv.first);
  }
  for (uint64_t k : gone) m->index.erase(k);
  return (int64_t)gone.size();
}

// Lookup count and last counting step of hashed keys (0, 0 for an absent key).
void orc_key_stats(void* h, const uint64_t* keys, int64_t n, uint64_t* freq, int64_t* last) {
  Model* m = (Model*)h;
  for (int64_t q = 0; q < n; ++q) {
    auto it = m->index.find(keys[q]);
    freq[q] = it == m->index.end() ? 0 : m->freq[it->second];
    last[q] = it == m->index.end() ? 0 : m->last_step[it->second];
  }
}

// Read parameters.  keys: global rows (static) or raw keys (hashed).
// w: [n][D], acc: [n][acc width], mag_w: [n][D] / mag_acc: [n][acc width] magnitudes of the
// update that last wrote each element (0 for a row never updated), found: [n] (static rows always "found": an untouched row
// is its initial value).  Any output pointer may be NULL.
void orc_read_rows(void* h, const uint64_t* keys, int64_t n, float* w, float* acc,
                   double* mag_w, double* mag_acc, int8_t* found) {
  Model* m = (Model*)h;
  const int D = m->D, AW = m->acc_width();
  for (int64_t q = 0; q < n; ++q) {
    auto it = m->index.find(keys[q]);
    if (it != m->index.end()) {
      const int64_t r = it->second;
      if (w) std::memcpy(w + q * D, &m->w[(size_t)r * D], sizeof(float) * D);
      if (acc) std::memcpy(acc + q * AW, &m->acc[(size_t)r * AW], sizeof(float) * AW);
      if (mag_w) std::memcpy(mag_w + q * D, &m->mag_w[(size_t)r * D], sizeof(double) * D);
      if (mag_acc) std::memcpy(mag_acc + q * AW, &m->mag_acc[(size_t)r * AW], sizeof(double) * AW);
      if (found) found[q] = 1;
      continue;
    }
    if (m->hashed) {
      if (found) found[q] = 0;
      continue;
    }
    const int64_t t = m->table_of_row(keys[q]);
    const int64_t id = (int64_t)keys[q] - m->base[t];
    for (int c = 0; c < D && w; ++c) {
      const float v = init_value(m->seed, (int)t, id, c, m->lo, m->hi);
      w[q * D + c] = m->bf16 ? bf16_to_float(bf16_rne(v)) : v;
    }
    for (int c = 0; c < AW && acc; ++c) acc[q * AW + c] = m->init_acc;
    for (int c = 0; c < D && mag_w; ++c) mag_w[q * D + c] = 0.0;
    for (int c = 0; c < AW && mag_acc; ++c) mag_acc[q * AW + c] = 0.0;
    if (found) found[q] = 1;
  }
}

// Unique keys of the last forward's valid lookups, ascending, with occurrence counts.
// Writes at most `cap` entries; returns the number of unique keys.
int64_t orc_unique(void* h, uint64_t* keys, int64_t* counts, int64_t cap) {
  Model* m = (Model*)h;
  std::map<uint64_t, int64_t> cnt;
  for (uint64_t k : m->lk_key) cnt[k] += 1;
  int64_t n = 0;
  for (auto& kv : cnt) {
    if (n < cap) {
      if (keys) keys[n] = kv.first;
      if (counts) counts[n] = kv.second;
    }
    ++n;
  }
  return n;
}

// Every materialised row (static: touched rows; hashed: inserted keys), ascending by key.
int64_t orc_export(void* h, uint64_t* keys, float* w, float* acc, int64_t cap) {
  Model* m = (Model*)h;
  std::vector<std::pair<uint64_t, int64_t>> all(m->index.begin(), m->index.end());
  std::sort(all.begin(), all.end());
  const int D = m->D, AW = m->acc_width();
  int64_t n = 0;
  for (auto& kv : all) {
    if (n < cap) {
      if (keys) keys[n] = kv.first;
      if (w) std::memcpy(w + n * D, &m->w[(size_t)kv.second * D], sizeof(float) * D);
      if (acc) std::memcpy(acc + n * AW, &m->acc[(size_t)kv.second * AW], sizeof(float) * AW);
    }
    ++n;
  }
  return n;
}

}  // extern "C"
