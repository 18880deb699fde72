// ggrn_oracle.cpp -- plain single-threaded CPU oracle of the fused gated
// group-RMSNorm.  TEST INFRASTRUCTURE ONLY (see ggrn_oracle.h): the product
// path never links or calls it.
//
// Build with -ffp-contract=off and without fast-math so that every f32
// operation below rounds once, on every host architecture.
#include "ggrn_oracle.h"

#include <cmath>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// T <-> f32 codecs, written from the IEEE-754 binary16 and bfloat16 bit
// layouts.  bfloat16 = the upper 16 bits of a binary32; binary16 = 1 sign
// bit, 5 exponent bits (bias 15), 10 fraction bits.  Both round to nearest,
// ties to even.
// ---------------------------------------------------------------------------
uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}
float bits_f32(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint16_t bf16_from_f32(float f) {
  uint32_t u = f32_bits(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) {            // NaN: keep sign and top payload, force quiet
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  }
  // Round to nearest even on the 16 dropped bits.  Overflow carries into the
  // exponent and lands on +-inf, which is the RNE result.
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

float bf16_to_f32(uint16_t h) { return bits_f32(static_cast<uint32_t>(h) << 16); }

uint16_t f16_from_f32(float f) {
  uint32_t u = f32_bits(f);
  uint16_t sign = static_cast<uint16_t>((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7fffffffu;
  if (a > 0x7f800000u) {                             // NaN
    return static_cast<uint16_t>(sign | 0x7e00u | ((a >> 13) & 0x03ffu));
  }
  if (a == 0x7f800000u) return static_cast<uint16_t>(sign | 0x7c00u);
  int e = static_cast<int>(a >> 23) - 127;           // unbiased binary32 exponent
  uint32_t mant = a & 0x007fffffu;
  if ((a >> 23) != 0) mant |= 0x00800000u;           // implicit bit (24-bit significand)
  else e = -126;                                     // binary32 subnormal
  if (e > 15) return static_cast<uint16_t>(sign | 0x7c00u);
  if (e >= -14) {
    // Normal binary16: keep 11 significand bits, drop 13.
    uint32_t m = mant >> 13;
    uint32_t rem = mant & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (m & 1u))) ++m;
    uint32_t he = static_cast<uint32_t>(e + 15);
    if (m == 0x800u) {  // significand overflow: next binade
      m = 0x400u;
      ++he;
    }
    if (he >= 31u) return static_cast<uint16_t>(sign | 0x7c00u);
    return static_cast<uint16_t>(sign | (he << 10) | (m & 0x03ffu));
  }
  // Subnormal binary16: value / 2^-24 = mant * 2^(e + 1).
  int shift = -(e + 1);  // >= 14
  if (shift > 25) return sign;  // below half the smallest subnormal
  uint32_t m = mant >> shift;
  uint32_t rem = mant & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (m & 1u))) ++m;
  // m == 0x400 is the smallest normal, which the same bit pattern encodes.
  return static_cast<uint16_t>(sign | m);
}

float f16_to_f32(uint16_t h) {
  uint32_t sign = (static_cast<uint32_t>(h) & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1fu;
  uint32_t m = h & 0x03ffu;
  float mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<float>(m), -24);                 // subnormal or zero
  } else if (e == 31) {
    return bits_f32(sign | 0x7f800000u | (m << 13) | (m ? 0x00400000u : 0u));
  } else {
    mag = std::ldexp(static_cast<float>(m | 0x400u), static_cast<int>(e) - 25);
  }
  return bits_f32(sign | f32_bits(mag));
}

// Round a double to the nearest T value (ties to even), directly, so the
// double twin does not round twice through f32.  Returns the rounded value
// as a double that T represents exactly (or +-inf / NaN).
double round_double_to(double v, int dtype) {
  if (dtype == GGRN_ORACLE_F32) return static_cast<double>(static_cast<float>(v));
  if (std::isnan(v) || std::isinf(v) || v == 0.0) return v;
  const int sig_bits = (dtype == GGRN_ORACLE_BF16) ? 8 : 11;    // significand incl. implicit bit
  const int min_exp = (dtype == GGRN_ORACLE_BF16) ? -126 : -14;  // smallest normal exponent
  const double max_finite = (dtype == GGRN_ORACLE_BF16)
                                ? std::ldexp(255.0, 120)          // (2 - 2^-7) * 2^127
                                : 65504.0;
  int e;
  std::frexp(v, &e);  // |v| in [2^(e-1), 2^e)
  int exp2 = e - 1;
  if (exp2 < min_exp) exp2 = min_exp;          // subnormal quantum
  const double q = std::ldexp(1.0, exp2 - (sig_bits - 1));
  double r = std::nearbyint(v / q) * q;        // exact scaling; default rounding is RNE
  if (std::fabs(r) > max_finite) r = std::copysign(INFINITY, v);
  return r;
}

// Typed element access.
float load_elem(const void* base, int64_t idx, int dtype) {
  if (dtype == GGRN_ORACLE_F32) return static_cast<const float*>(base)[idx];
  uint16_t h = static_cast<const uint16_t*>(base)[idx];
  return dtype == GGRN_ORACLE_BF16 ? bf16_to_f32(h) : f16_to_f32(h);
}

// Round f32 -> T and return the T value widened back to f32.
float round_to_t(float v, int dtype) {
  if (dtype == GGRN_ORACLE_F32) return v;
  if (dtype == GGRN_ORACLE_BF16) return bf16_to_f32(bf16_from_f32(v));
  return f16_to_f32(f16_from_f32(v));
}

// Store an f32 value as T (RNE).
void store_elem(void* base, int64_t idx, float v, int dtype) {
  if (dtype == GGRN_ORACLE_F32) {
    static_cast<float*>(base)[idx] = v;
  } else if (dtype == GGRN_ORACLE_BF16) {
    static_cast<uint16_t*>(base)[idx] = bf16_from_f32(v);
  } else {
    static_cast<uint16_t*>(base)[idx] = f16_from_f32(v);
  }
}

// Store a double that T represents exactly (output of round_double_to).
void store_exact(void* base, int64_t idx, double v, int dtype) {
  store_elem(base, idx, static_cast<float>(v), dtype);
}

// silu(x) = x * sigmoid(x) = x / (1 + exp(-x)), in f32.
float silu_f32(float x) { return x / (1.0f + std::exp(-x)); }

double silu_f64(double x) { return x / (1.0 + std::exp(-x)); }

int validate(const void* y, const void* gate, const void* w, const void* out,
             int64_t rows, int64_t width, int64_t gs, int64_t ys, int64_t gts,
             int64_t os, int dtype, int mode) {
  if (dtype != GGRN_ORACLE_F32 && dtype != GGRN_ORACLE_F16 && dtype != GGRN_ORACLE_BF16)
    return GGRN_ORACLE_ERR_DTYPE;
  if (mode != GGRN_ORACLE_MODE_MAMBA2 && mode != GGRN_ORACLE_MODE_ONNX)
    return GGRN_ORACLE_ERR_DTYPE;
  // The ONNX contract admits float32 and float16 only.
  if (mode == GGRN_ORACLE_MODE_ONNX && dtype == GGRN_ORACLE_BF16) return GGRN_ORACLE_ERR_DTYPE;
  if (rows < 0 || width <= 0 || gs <= 0 || width % gs != 0) return GGRN_ORACLE_ERR_SHAPE;
  if (rows > 0 && (ys < width || gts < width || os < width)) return GGRN_ORACLE_ERR_SHAPE;
  if (rows > 0 && (!y || !gate || !w || !out)) return GGRN_ORACLE_ERR_NULL;
  return GGRN_ORACLE_OK;
}

}  // namespace

extern "C" int ggrn_oracle_forward_pre(const void* y, const void* gate, const void* w,
                                       void* out, void* t_out, float* pre_out, int64_t rows,
                                       int64_t width, int64_t group_size,
                                       int64_t y_row_stride, int64_t gate_row_stride,
                                       int64_t out_row_stride, float eps, int dtype,
                                       int mode) {
  int st = validate(y, gate, w, out, rows, width, group_size, y_row_stride,
                    gate_row_stride, out_row_stride, dtype, mode);
  if (st != GGRN_ORACLE_OK || rows == 0) return st;

  const int64_t gs = group_size;
  const int64_t groups = width / gs;
  const float gs_f = static_cast<float>(gs);
  std::vector<float> gated(static_cast<size_t>(gs));
  std::vector<float> x(static_cast<size_t>(gs));

  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t g = 0; g < groups; ++g) {
      const int64_t col0 = g * gs;
      float m2 = 0.0f;
      if (mode == GGRN_ORACLE_MODE_MAMBA2) {
        // gated = f32(y) * silu(f32(gate))
        for (int64_t j = 0; j < gs; ++j) {
          float a = load_elem(y, n * y_row_stride + col0 + j, dtype);
          float b = load_elem(gate, n * gate_row_stride + col0 + j, dtype);
          gated[j] = a * silu_f32(b);
        }
        // m2 = sum_j gated^2, sequential in j
        for (int64_t j = 0; j < gs; ++j) {
          float sq = gated[j] * gated[j];
          m2 = m2 + sq;
        }
      } else {
        // mean(X^2) over the group
        for (int64_t j = 0; j < gs; ++j) {
          x[j] = load_elem(y, n * y_row_stride + col0 + j, dtype);
          float sq = x[j] * x[j];
          m2 = m2 + sq;
        }
      }
      // nf = rsqrt(m2 / group_size + eps)
      float v = m2 / gs_f;
      v = v + eps;
      const float nf = static_cast<float>(1.0 / std::sqrt(static_cast<double>(v)));

      for (int64_t j = 0; j < gs; ++j) {
        const int64_t col = col0 + j;
        if (mode == GGRN_ORACLE_MODE_MAMBA2) {
          // out = cast(f32(w[col]) * f32(cast(gated * nf, T)), T)
          const float pre = gated[j] * nf;
          if (pre_out) pre_out[n * width + col] = pre;
          float t = round_to_t(pre, dtype);
          if (t_out) store_elem(t_out, n * width + col, t, dtype);
          float p = static_cast<const float*>(w)[col] * t;
          store_elem(out, n * out_row_stride + col, p, dtype);
        } else {
          // Y = X * nf * scale * SiLU(gate), f32 until the store
          float b = load_elem(gate, n * gate_row_stride + col, dtype);
          float s = load_elem(w, j, dtype);
          float r = x[j] * nf;
          r = r * s;
          r = r * silu_f32(b);
          if (pre_out) pre_out[n * width + col] = r;
          store_elem(out, n * out_row_stride + col, r, dtype);
        }
      }
    }
  }
  return GGRN_ORACLE_OK;
}

extern "C" int ggrn_oracle_forward_ex(const void* y, const void* gate, const void* w,
                                      void* out, void* t_out, int64_t rows,
                                      int64_t width, int64_t group_size,
                                      int64_t y_row_stride, int64_t gate_row_stride,
                                      int64_t out_row_stride, float eps, int dtype,
                                      int mode) {
  return ggrn_oracle_forward_pre(y, gate, w, out, t_out, nullptr, rows, width, group_size,
                                 y_row_stride, gate_row_stride, out_row_stride, eps, dtype,
                                 mode);
}

extern "C" int ggrn_oracle_forward(const void* y, const void* gate, const void* w, void* out,
                                   int64_t rows, int64_t width, int64_t group_size,
                                   int64_t y_row_stride, int64_t gate_row_stride,
                                   int64_t out_row_stride, float eps, int dtype, int mode) {
  return ggrn_oracle_forward_ex(y, gate, w, out, nullptr, rows, width, group_size,
                                y_row_stride, gate_row_stride, out_row_stride, eps, dtype,
                                mode);
}

extern "C" int ggrn_oracle_forward_f64(const void* y, const void* gate, const void* w,
                                       void* out, int64_t rows, int64_t width,
                                       int64_t group_size, int64_t y_row_stride,
                                       int64_t gate_row_stride, int64_t out_row_stride,
                                       float eps, int dtype, int mode) {
  int st = validate(y, gate, w, out, rows, width, group_size, y_row_stride,
                    gate_row_stride, out_row_stride, dtype, mode);
  if (st != GGRN_ORACLE_OK || rows == 0) return st;

  const int64_t gs = group_size;
  const int64_t groups = width / gs;
  std::vector<double> a(static_cast<size_t>(gs));
  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t g = 0; g < groups; ++g) {
      const int64_t col0 = g * gs;
      double m2 = 0.0;
      for (int64_t j = 0; j < gs; ++j) {
        double yv = load_elem(y, n * y_row_stride + col0 + j, dtype);
        if (mode == GGRN_ORACLE_MODE_MAMBA2) {
          double b = load_elem(gate, n * gate_row_stride + col0 + j, dtype);
          a[j] = yv * silu_f64(b);
        } else {
          a[j] = yv;
        }
        m2 += a[j] * a[j];
      }
      const double nf = 1.0 / std::sqrt(m2 / static_cast<double>(gs) + static_cast<double>(eps));
      for (int64_t j = 0; j < gs; ++j) {
        const int64_t col = col0 + j;
        double r;
        if (mode == GGRN_ORACLE_MODE_MAMBA2) {
          double t = round_double_to(a[j] * nf, dtype);
          r = round_double_to(static_cast<double>(static_cast<const float*>(w)[col]) * t, dtype);
        } else {
          double b = load_elem(gate, n * gate_row_stride + col, dtype);
          double s = load_elem(w, j, dtype);
          r = round_double_to(a[j] * nf * s * silu_f64(b), dtype);
        }
        store_exact(out, n * out_row_stride + col, r, dtype);
      }
    }
  }
  return GGRN_ORACLE_OK;
}

extern "C" void ggrn_oracle_encode(const float* in, void* out, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) store_elem(out, i, in[i], dtype);
}

extern "C" void ggrn_oracle_decode(const void* in, float* out, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) out[i] = load_elem(in, i, dtype);
}
