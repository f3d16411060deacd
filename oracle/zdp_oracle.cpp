// zdp_oracle.cpp -- plain, slow, single-threaded CPU oracle for the ZeRO
// synchronisation-and-update step.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product links, loads or calls this
// file.  It exists so that tests, the smoke check and the benchmark's CPU
// baseline can check the CUDA library against an independent statement of
// what the step computes.  It shares no code, header, table or constant with
// the CUDA path.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.
// -ffp-contract=off matters: aarch64 GCC fuses a*b+c into one FMA by default,
// and every formula below is meant to round after each operation.
//
// Sources (the pages, by title and section):
//  [F9]  Fudan MLSys, ch. 9 "Distributed training and data parallelism":
//        9.2.2 (Adam), 9.3.5 (collectives), 9.3.6 (ring all-reduce),
//        9.4.2 (ZeRO, 16 bytes per parameter).
//  [L7]  CS336 Lecture 7 notes, "Parallelism I - collectives, data
//        parallelism and ZeRO": 3.4 (all-reduce = reduce-scatter +
//        all-gather), 4.2 (ring algorithm and its p=4 trace), 4.3 (volume),
//        6.2 (all_reduce SUM then divide by world size), 7 (16 B/param),
//        8.1 (FlatZeRO1), 11 (exercises 1, 2, 6).
//  [IG]  "Must-know: communication cost of LLM training" interview guide,
//        1.4 item 6 (reduce-scatter: GPU r receives reduced chunk r),
//        2.4 (ring volume 2(N-1)/N).
//
// Readings where the pages are silent (each also listed in the design notes):
//  * rank r owns flat chunk r = [r*S, (r+1)*S), S = ceil(n/P), zero padding
//    at the tail ([L7] 11 exercise 1(e); [IG] 1.4 item 6);
//  * the ring sum for chunk r starts at rank (r+1) mod P and ends with rank r's
//    own value, accumulating in fp32 ([F9] 9.3.6; [L7] 4.2 relabelled so that
//    the rank holding a finished chunk is its owner);
//  * averaging is one multiply by `scale` after the full sum ([L7] 6.2);
//  * AdamW = the Adam of [F9] 9.2.2 plus decoupled weight decay applied to
//    the pre-update weight: w <- w - (lr*wd)*w - lr*u;
//  * bias corrections 1 - beta^t are evaluated in double and rounded to fp32;
//  * fp32 -> bf16 is round-to-nearest-even; NaN becomes a quiet NaN;
//  * ZeRO++ ([F9] 9.4.3: weights quantized to INT8 before the all-gather and
//    dequantized after it; gradients quantized block-wise for the
//    reduce-scatter): blocks of 256 consecutive elements (global index i in
//    block i / 256); scale = max|x| / 127 over the block (fp32 division),
//    q = x / scale rounded half to even and clamped to [-127, 127]; an
//    all-zero block has scale 0 and q = 0; dequantization is q * scale in
//    fp32.  (Not on the page, a reading: a block holding a NaN has a NaN
//    scale, one holding an infinity an infinite scale, and a NaN quotient is
//    clamped to -127, so that such a block dequantizes to non-finite values
//    and the overflow flag reports it.)  The quantized all-gather quantizes the bf16 parameter; a
//    quantized gradient is dequantized in fp32 before the ring sum;
//  * with bf16 moments (CS336 Lecture 7 notes, 8.4: everything but the fp32
//    master weight in BF16, 12 bytes per parameter) m and v are stored in
//    bf16: widened exactly when loaded, updated in fp32, the update uses the
//    fresh fp32 moments, and they are rounded to nearest even when stored.

#include <algorithm>
#include <cmath>
#include <limits>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Number formats, from the IEEE-754 binary16 / binary32 definitions and the
// bfloat16 definition (the upper 16 bits of a binary32).
// ---------------------------------------------------------------------------

float bits_to_float(uint32_t u) {
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

uint32_t float_to_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return u;
}

// bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits
// of a binary32, so widening is exact: put the 16 bits on top.
float bf16_to_float(uint16_t h) { return bits_to_float(static_cast<uint32_t>(h) << 16); }

// binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
float fp16_to_float(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  float mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<float>(f), -24);  // subnormal: f * 2^-24
  } else if (e == 31) {
    if (f == 0) {
      mag = INFINITY;
    } else {
      // NaN: keep the payload in the top fraction bits, as a widening does.
      uint32_t u = 0x7f800000u | (static_cast<uint32_t>(f) << 13);
      mag = bits_to_float(u);
    }
  } else {
    mag = std::ldexp(static_cast<float>(1024 + f), e - 25);  // (1 + f/1024) * 2^(e-15)
  }
  return sign ? -mag : mag;
}

float widen(uint16_t h, int gdt) { return gdt == 0 ? bf16_to_float(h) : fp16_to_float(h); }

// fp32 -> bf16, round to nearest, ties to even.  For a finite value the two
// candidate bf16 numbers are the truncation `lo` and its successor `lo + 1`
// (bit patterns of same-signed floats are ordered like their magnitudes, and
// the carry out of the fraction moves to the next binade or to infinity, as
// it should).  The dropped 16 bits decide: above half -> up, below -> down,
// exactly half -> whichever candidate has an even last bit.
uint16_t float_to_bf16_rne(float x) {
  const uint32_t u = float_to_bits(x);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0) {
    return static_cast<uint16_t>(((u >> 16) & 0x8000u) | 0x7fc0u);  // quiet NaN
  }
  uint32_t lo = u >> 16;
  const uint32_t rest = u & 0xffffu;
  if (rest > 0x8000u || (rest == 0x8000u && (lo & 1u))) lo += 1;
  return static_cast<uint16_t>(lo);
}

bool is_finite(float x) { return (float_to_bits(x) & 0x7f800000u) != 0x7f800000u; }

// ---------------------------------------------------------------------------
// Ownership: S = ceil(n/P); rank r owns [r*S, (r+1)*S).
// ---------------------------------------------------------------------------

int64_t shard_size(int64_t n, int P) { return (n + P - 1) / P; }

int owner_of(int64_t i, int64_t S) { return static_cast<int>(i / S); }

// Ring-order sum of the P ranks' values of one element owned by rank r:
// start with rank (r+1) mod P, then add ranks (r+2) mod P, ..., r.
// `vals[q]` is rank q's widened value.
float ring_sum(const float* vals, int P, int r) {
  float acc = vals[(r + 1) % P];
  for (int k = 2; k <= P; ++k) acc = acc + vals[(r + k) % P];
  return acc;
}

// ---------------------------------------------------------------------------
// AdamW on one element ([F9] 9.2.2 plus decoupled decay).
// ---------------------------------------------------------------------------

struct Adam {
  float lr, b1, b2, eps, one_minus_b1, one_minus_b2, lr_wd, bc1, bc2;
};

Adam make_adam(float lr, float b1, float b2, float eps, float wd, int t) {
  Adam a;
  a.lr = lr;
  a.b1 = b1;
  a.b2 = b2;
  a.eps = eps;
  a.one_minus_b1 = 1.0f - b1;
  a.one_minus_b2 = 1.0f - b2;
  a.lr_wd = lr * wd;
  a.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(t)));
  a.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2), static_cast<double>(t)));
  return a;
}

// m_t = b1 m + (1-b1) g ; v_t = b2 v + (1-b2) g^2 ;
// m_hat = m_t / (1 - b1^t) ; v_hat = v_t / (1 - b2^t) ;
// w <- w - lr*wd*w - lr * m_hat / (sqrt(v_hat) + eps).
void adamw_element(float& w, float& m, float& v, float g, const Adam& a) {
  const float m_new = a.b1 * m + a.one_minus_b1 * g;
  const float g_sq = g * g;
  const float v_new = a.b2 * v + a.one_minus_b2 * g_sq;
  const float m_hat = m_new / a.bc1;
  const float v_hat = v_new / a.bc2;
  const float denom = std::sqrt(v_hat) + a.eps;
  const float u = m_hat / denom;
  const float w_decayed = w - a.lr_wd * w;
  w = w_decayed - a.lr * u;
  m = m_new;
  v = v_new;
}

// ---------------------------------------------------------------------------
// Block-wise int8 quantization (ZeRO++, [F9] 9.4.3).
// ---------------------------------------------------------------------------
constexpr int64_t kQBlock = 256;

// The block's largest magnitude over 127.  A NaN anywhere in the block makes
// the maximum, and so the scale, NaN; an infinity (and no NaN) makes it
// infinite.  A non-finite block thus dequantizes to non-finite values.
float quant_scale(const float* x, int64_t count) {
  float amax = 0.0f;
  for (int64_t k = 0; k < count; ++k) {
    const float a = std::fabs(x[k]);
    if (std::isnan(a)) return std::numeric_limits<float>::quiet_NaN();
    if (a > amax) amax = a;
  }
  return amax / 127.0f;
}

int8_t quant_one(float x, float scale) {
  if (scale == 0.0f) return 0;
  const float y = x / scale;
  // x / NaN, or an infinity over an infinite scale: not a number, which the
  // clamp to [-127, 127] sends to its lower end.
  if (std::isnan(y)) return -127;
  float r = std::nearbyint(y);  // the default rounding mode: half to even
  if (r > 127.0f) r = 127.0f;
  if (r < -127.0f) r = -127.0f;
  return static_cast<int8_t>(r);
}

float dequant_one(int8_t q, float scale) { return static_cast<float>(q) * scale; }

// Moments stored as fp32 (mdt == 0) or bf16 bit patterns (mdt == 1).
float load_moment(const void* base, int64_t k, int mdt) {
  return mdt == 0 ? static_cast<const float*>(base)[k]
                  : bf16_to_float(static_cast<const uint16_t*>(base)[k]);
}

void store_moment(void* base, int64_t k, int mdt, float x) {
  if (mdt == 0) {
    static_cast<float*>(base)[k] = x;
  } else {
    static_cast<uint16_t*>(base)[k] = float_to_bf16_rne(x);
  }
}

}  // namespace

extern "C" {

// ---- formats --------------------------------------------------------------
float ora_bf16_to_f32(uint16_t h) { return bf16_to_float(h); }
float ora_f16_to_f32(uint16_t h) { return fp16_to_float(h); }
uint16_t ora_f32_to_bf16(float x) { return float_to_bf16_rne(x); }

void ora_bf16_to_f32_array(const uint16_t* in, float* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) out[i] = bf16_to_float(in[i]);
}
void ora_f16_to_f32_array(const uint16_t* in, float* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) out[i] = fp16_to_float(in[i]);
}
void ora_f32_to_bf16_array(const float* in, uint16_t* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) out[i] = float_to_bf16_rne(in[i]);
}

int64_t ora_shard_size(int64_t n, int P) { return shard_size(n, P); }

// ---- the ring, literally ---------------------------------------------------
// P ranks, each holding a buffer of P chunks of S fp32 values, laid out as
// bufs[rank*P*S + chunk*S + e].  Every step, every rank sends one chunk to
// rank+1 (mod P); all sends of a step are taken from the state before that
// step, then delivered.  `sent[rank]` counts elements sent.
//
// Reduce-scatter step s: rank i sends chunk (i - s - shift) mod P, and the
// receiver adds it into its own copy of that chunk.  With shift = 0 this is
// the schedule printed in [L7] 4.2 (rank i finishes with chunk i+1); with
// shift = 1, rank i finishes with chunk i, its own.
void ora_ring_reduce_scatter_sim(float* bufs, int P, int64_t S, int shift, int64_t* sent) {
  const int64_t row = static_cast<int64_t>(P) * S;
  std::vector<float> msg(static_cast<size_t>(row));  // one message slot of S per sender
  std::vector<int> chunk(P);
  for (int s = 0; s < P - 1; ++s) {
    for (int i = 0; i < P; ++i) {
      int c = ((i - s - shift) % P + P) % P;
      chunk[i] = c;
      for (int64_t e = 0; e < S; ++e) msg[i * S + e] = bufs[i * row + c * S + e];
      sent[i] += S;
    }
    for (int i = 0; i < P; ++i) {
      const int dst = (i + 1) % P;
      const int c = chunk[i];
      for (int64_t e = 0; e < S; ++e) {
        float& mine = bufs[dst * row + c * S + e];
        mine = msg[i * S + e] + mine;  // received partial sum + own chunk
      }
    }
  }
}

// All-gather step s: rank i forwards chunk (i + 1 - shift - s) mod P, the one
// it finished (s = 0) or received in the previous step; the receiver
// overwrites its copy.
void ora_ring_all_gather_sim(float* bufs, int P, int64_t S, int shift, int64_t* sent) {
  const int64_t row = static_cast<int64_t>(P) * S;
  std::vector<float> msg(static_cast<size_t>(row));
  std::vector<int> chunk(P);
  for (int s = 0; s < P - 1; ++s) {
    for (int i = 0; i < P; ++i) {
      int c = ((i + 1 - shift - s) % P + P) % P;
      chunk[i] = c;
      for (int64_t e = 0; e < S; ++e) msg[i * S + e] = bufs[i * row + c * S + e];
      sent[i] += S;
    }
    for (int i = 0; i < P; ++i) {
      const int dst = (i + 1) % P;
      const int c = chunk[i];
      for (int64_t e = 0; e < S; ++e) bufs[dst * row + c * S + e] = msg[i * S + e];
    }
  }
}

// ---- the collectives by definition -------------------------------------------
// grads: P rows with row stride `ld` elements; row q holds rank q's gradient
// of elements [0, n) (bf16 if gdt == 0, fp16 if gdt == 1).
// shards: P*S fp32.  shards[i] = ring sum of element i times `scale` for
// i < n, and 0 for the padding i in [n, P*S).  The overflow word is OR-ed with
// 1 if any reduced value is not finite; sumsq (if not null) gets the fp64 sum
// of squares of the reduced values added to it, in element order.
void ora_reduce_scatter(const uint16_t* grads, int64_t ld, int gdt, float* shards, int64_t n,
                        int P, float scale, int32_t* overflow, double* sumsq) {
  const int64_t S = shard_size(n, P);
  std::vector<float> vals(P);
  int32_t flag = 0;
  double ss = 0.0;
  for (int64_t i = 0; i < static_cast<int64_t>(P) * S; ++i) {
    if (i >= n) {
      shards[i] = 0.0f;
      continue;
    }
    for (int q = 0; q < P; ++q) vals[q] = widen(grads[q * ld + i], gdt);
    const float g = ring_sum(vals.data(), P, owner_of(i, S)) * scale;
    if (!is_finite(g)) flag = 1;
    ss += static_cast<double>(g) * static_cast<double>(g);
    shards[i] = g;
  }
  if (overflow) *overflow |= flag;
  if (sumsq) *sumsq += ss;
}

// Elementwise AdamW over `count` elements of one shard.
void ora_adamw(float* w, float* m, float* v, const float* g, int64_t count, float lr, float b1,
               float b2, float eps, float wd, int t) {
  const Adam a = make_adam(lr, b1, b2, eps, wd, t);
  for (int64_t i = 0; i < count; ++i) adamw_element(w[i], m[i], v[i], g[i], a);
}

// All-gather of the updated parameters: every replica row receives the bf16
// (round-to-nearest-even) value of master[i], for i < n.
void ora_all_gather(const float* master, uint16_t* replicas, int64_t rld, int64_t n, int P) {
  for (int q = 0; q < P; ++q)
    for (int64_t i = 0; i < n; ++i) replicas[q * rld + i] = float_to_bf16_rne(master[i]);
}

// ---- the fused step by definition -------------------------------------------
// Processes the global element range [off, off+len) of an n-element model.
// grads row q (stride ld) holds rank q's gradient for that range: element
// off+j is grads[q*ld + j].  master/m/v hold global elements from `base` on:
// element i is master[i - base]; replica row q (stride rld) likewise.  With
// check_overflow != 0 and a non-finite reduced gradient anywhere in the
// range, nothing is written.  Returns 0, or -1 on bad arguments.
int ora_step_mdt(const uint16_t* grads, int64_t ld, int gdt, float* master, void* m, void* v,
                 int mdt, uint16_t* replicas, int64_t rld, int64_t base, int64_t n, int64_t off,
                 int64_t len, int P, float scale, float lr, float b1, float b2, float eps,
                 float wd, int t, int check_overflow, int32_t* overflow, double* sumsq) {
  if (P < 1 || n < 1 || off < 0 || len < 0 || off + len > n || t < 1 || base > off ||
      (mdt != 0 && mdt != 1))
    return -1;
  const int64_t S = shard_size(n, P);
  const Adam a = make_adam(lr, b1, b2, eps, wd, t);
  std::vector<float> vals(P);
  std::vector<float> g(static_cast<size_t>(len));
  int32_t flag = 0;
  double ss = 0.0;
  for (int64_t j = 0; j < len; ++j) {
    const int64_t i = off + j;
    for (int q = 0; q < P; ++q) vals[q] = widen(grads[q * ld + j], gdt);
    g[j] = ring_sum(vals.data(), P, owner_of(i, S)) * scale;
    if (!is_finite(g[j])) flag = 1;
    ss += static_cast<double>(g[j]) * static_cast<double>(g[j]);
  }
  if (overflow) *overflow |= flag;
  if (sumsq) *sumsq += ss;
  if (check_overflow && flag) return 0;
  for (int64_t j = 0; j < len; ++j) {
    const int64_t k = off + j - base;
    float mk = load_moment(m, k, mdt), vk = load_moment(v, k, mdt);
    adamw_element(master[k], mk, vk, g[j], a);
    store_moment(m, k, mdt, mk);
    store_moment(v, k, mdt, vk);
    const uint16_t p = float_to_bf16_rne(master[k]);
    for (int q = 0; q < P; ++q) replicas[q * rld + k] = p;
  }
  return 0;
}

// The step with fp32 moments.
int ora_step(const uint16_t* grads, int64_t ld, int gdt, float* master, float* m, float* v,
             uint16_t* replicas, int64_t rld, int64_t base, int64_t n, int64_t off, int64_t len,
             int P, float scale, float lr, float b1, float b2, float eps, float wd, int t,
             int check_overflow, int32_t* overflow, double* sumsq) {
  return ora_step_mdt(grads, ld, gdt, master, m, v, 0, replicas, rld, base, n, off, len, P, scale,
                      lr, b1, b2, eps, wd, t, check_overflow, overflow, sumsq);
}

// The same step on a sample of k elements given by their global indices
// idx[0..k).  gs row q (stride k) holds rank q's gradient at those indices;
// w/m/v are the state values there and are updated in place unless `skip`;
// gout receives the reduced gradient and rep the bf16 value every replica
// must hold.  `skip` is the caller's skip decision for the whole step.
int ora_step_sampled_mdt(const uint16_t* gs, const int64_t* idx, int64_t k, int gdt, float* w,
                         void* m, void* v, int mdt, float* gout, uint16_t* rep, int64_t n, int P,
                         float scale, float lr, float b1, float b2, float eps, float wd, int t,
                         int skip, int32_t* overflow) {
  if (P < 1 || n < 1 || t < 1 || (mdt != 0 && mdt != 1)) return -1;
  const int64_t S = shard_size(n, P);
  const Adam a = make_adam(lr, b1, b2, eps, wd, t);
  std::vector<float> vals(P);
  int32_t flag = 0;
  for (int64_t j = 0; j < k; ++j) {
    if (idx[j] < 0 || idx[j] >= n) return -1;
    for (int q = 0; q < P; ++q) vals[q] = widen(gs[q * k + j], gdt);
    const float g = ring_sum(vals.data(), P, owner_of(idx[j], S)) * scale;
    if (!is_finite(g)) flag = 1;
    gout[j] = g;
    if (!skip) {
      float mj = load_moment(m, j, mdt), vj = load_moment(v, j, mdt);
      adamw_element(w[j], mj, vj, g, a);
      store_moment(m, j, mdt, mj);
      store_moment(v, j, mdt, vj);
    }
    rep[j] = float_to_bf16_rne(w[j]);
  }
  if (overflow) *overflow |= flag;
  return 0;
}

int ora_step_sampled(const uint16_t* gs, const int64_t* idx, int64_t k, int gdt, float* w,
                     float* m, float* v, float* gout, uint16_t* rep, int64_t n, int P, float scale,
                     float lr, float b1, float b2, float eps, float wd, int t, int skip,
                     int32_t* overflow) {
  return ora_step_sampled_mdt(gs, idx, k, gdt, w, m, v, 0, gout, rep, n, P, scale, lr, b1, b2,
                              eps, wd, t, skip, overflow);
}

// ---- ZeRO++ block quantization -----------------------------------------------
// x[0..n) -> q[0..n), scales[0..ceil(n/256)): block b covers [256b, 256b+256).
void ora_quantize_blocks(const float* x, int64_t n, int8_t* q, float* scales) {
  for (int64_t b = 0; b * kQBlock < n; ++b) {
    const int64_t lo = b * kQBlock, cnt = std::min<int64_t>(kQBlock, n - lo);
    scales[b] = quant_scale(x + lo, cnt);
    for (int64_t k = 0; k < cnt; ++k) q[lo + k] = quant_one(x[lo + k], scales[b]);
  }
}

void ora_dequantize_blocks(const int8_t* q, const float* scales, int64_t n, float* x) {
  for (int64_t i = 0; i < n; ++i) x[i] = dequant_one(q[i], scales[i / kQBlock]);
}

// The ZeRO++ step over the global range [off, off+len) of an n-element model
// (off a multiple of 256; off+len a multiple of 256 or n).  Rank q's gradient
// of element off+j is the int8 gq[q*ld + j] times the fp32 scale
// gs[q*sld + (off+j)/256 - off/256]; master/m/v hold global elements from
// `base` on (m/v fp32 or bf16 per mdt); rank q's replica of element i is the
// int8 rq[q*rld + i - base] with scale rs[q*rsld + i/256 - base/256] (base a
// multiple of 256), quantized from the bf16 parameter.  No overflow skip.
int ora_step_zpp(const int8_t* gq, int64_t ld, const float* gs, int64_t sld, float* master,
                 void* m, void* v, int mdt, int8_t* rq, int64_t rld, float* rs, int64_t rsld,
                 int64_t base, int64_t n, int64_t off, int64_t len, int P, float scale, float lr,
                 float b1, float b2, float eps, float wd, int t, int32_t* overflow,
                 double* sumsq) {
  if (P < 1 || n < 1 || off < 0 || len < 0 || off + len > n || t < 1 || base > off ||
      off % kQBlock != 0 || base % kQBlock != 0 || ((off + len) % kQBlock != 0 && off + len != n) ||
      (mdt != 0 && mdt != 1))
    return -1;
  const int64_t S = shard_size(n, P);
  const Adam a = make_adam(lr, b1, b2, eps, wd, t);
  std::vector<float> vals(P);
  std::vector<float> p(static_cast<size_t>(len));
  int32_t flag = 0;
  double ss = 0.0;
  for (int64_t j = 0; j < len; ++j) {
    const int64_t i = off + j;
    for (int q = 0; q < P; ++q)
      vals[q] = dequant_one(gq[q * ld + j], gs[q * sld + i / kQBlock - off / kQBlock]);
    const float g = ring_sum(vals.data(), P, owner_of(i, S)) * scale;
    if (!is_finite(g)) flag = 1;
    ss += static_cast<double>(g) * static_cast<double>(g);
    const int64_t k = i - base;
    float mk = load_moment(m, k, mdt), vk = load_moment(v, k, mdt);
    adamw_element(master[k], mk, vk, g, a);
    store_moment(m, k, mdt, mk);
    store_moment(v, k, mdt, vk);
    p[j] = bf16_to_float(float_to_bf16_rne(master[k]));  // the bf16 parameter
  }
  if (overflow) *overflow |= flag;
  if (sumsq) *sumsq += ss;
  for (int64_t lo = 0; lo < len; lo += kQBlock) {
    const int64_t cnt = std::min<int64_t>(kQBlock, len - lo);
    const int64_t blk = (off + lo) / kQBlock - base / kQBlock;
    const float sc = quant_scale(p.data() + lo, cnt);
    for (int q = 0; q < P; ++q) {
      rs[q * rsld + blk] = sc;
      for (int64_t e = 0; e < cnt; ++e)
        rq[q * rld + off + lo + e - base] = quant_one(p[lo + e], sc);
    }
  }
  return 0;
}

}  // extern "C"
