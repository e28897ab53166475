// oracle.cpp — plain, slow, single-threaded CPU oracle of the BitDelta hot path.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
// the CPU-baseline leg of the benchmark load this library.  The product path
// (the CUDA library under bit_weight_delta_gb300/) never links, loads or calls
// it, and this file includes nothing from that library: no shared headers,
// helpers, tables or constants.
//
// Source of every formula: the web page "BitDelta: serving 14 Zen models from
// one GPU cluster" (hanzo blog, 2026-02-28).  Citations below name a section
// of that page:
//   [Math]    section "Mathematical foundation" (Landasan Matematika)
//   [Serving] section "Serving architecture" (Arsitektur Penyajian), including
//             its conceptual fused_bitdelta_linear listing
//   [Infra]   section "Infrastructure details" (Rincian Infrastruktur),
//             paragraph "delta storage format"
//
// Arithmetic: fp64 for every sum and product, except where the method's own
// result is a binary32 / bf16 value (alpha is stored as float32 [Infra]; the
// effective weight is rounded to the dtype of W_base [Serving]).  Build with
// -ffp-contract=off and without -ffast-math so every operation is one IEEE
// operation in the stated precision.
//
// Readings where the page is silent (each is listed in the design notes too):
//   * bit order inside a byte: bit j of byte k is column 8k+j (LSB first);
//     bit value 1 means +1 [Infra says only "8 bits per byte"].
//   * sign(0) = +1: a zero delta stores bit 1 [Math says only "positive or
//     negative"].
//   * alpha scope: per matrix [Math] or one per output row [Infra]; the
//     per-row alpha is the same mean-|delta| estimator restricted to the row.
//   * effective weight: W_eff = bf16_rne( fp32(W_base) + (bit ? a : -a) ),
//     the add in IEEE binary32, then round-to-nearest-even to bf16.
//   * linear: y[m][n] = sum_k x[m][k] * W_eff[n][k] (F.linear, no bias),
//     x flattened to [M, d_in]; variant 0 in the grouped form is the base
//     model, W_eff = W_base.
//
// Parity pins: every function is pinned by tests in tests/test_oracle_pins.py
// (hand-derived fixtures, closed forms, library routines, invariants).

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>

namespace {

// bf16 <-> binary32 (the oracle's own helpers).
float bf16_bits_to_float(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// Round a binary32 value to the nearest bf16, ties to even.  NaN inputs are
// outside the contract (no input generator produces them).
uint16_t float_to_bf16_bits_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

// Neumaier-compensated running sum in fp64.
struct CompensatedSum {
  double s = 0.0;
  double c = 0.0;
  void add(double v) {
    double t = s + v;
    if (std::fabs(s) >= std::fabs(v))
      c += (s - t) + v;
    else
      c += (v - t) + s;
    s = t;
  }
  double value() const { return s + c; }
};

// [Math] Δ = W_ft − W_base, elementwise.  Both operands are bf16 values, so
// the fp64 difference is exact.
double delta_at(const uint16_t* w_base, const uint16_t* w_ft, int64_t idx) {
  return static_cast<double>(bf16_bits_to_float(w_ft[idx])) -
         static_cast<double>(bf16_bits_to_float(w_base[idx]));
}

// [Math] sign(Δ) reduced to one bit; bit 1 stands for +1 and sign(0) = +1.
int sign_bit(const uint16_t* w_base, const uint16_t* w_ft, int64_t idx) {
  float ft = bf16_bits_to_float(w_ft[idx]);
  float b = bf16_bits_to_float(w_base[idx]);
  return (ft < b) ? 0 : 1;
}

// [Infra] unpack: the bit of column `col` in row `row` of the packed matrix.
int packed_bit(const uint8_t* packed, int64_t d_in, int64_t row, int64_t col) {
  const uint8_t byte = packed[row * (d_in / 8) + col / 8];
  return (byte >> (col % 8)) & 1;
}

float alpha_for_row(const float* alpha, int per_row, int64_t row) {
  return per_row ? alpha[row] : alpha[0];
}

// [Serving] W_eff = W_base + α·sign(Δ), one element, in the dtype of W_base.
uint16_t effective_weight(uint16_t w_base_bits, int bit, float a) {
  float signed_alpha = bit ? a : -a;
  float sum = bf16_bits_to_float(w_base_bits) + signed_alpha;  // binary32 add
  return float_to_bf16_bits_rne(sum);
}

}  // namespace

extern "C" {

// [Infra] packed storage: 8 sign bits per byte, [d_out, d_in/8].
int64_t orc_packed_bytes(int64_t d_out, int64_t d_in) { return d_out * (d_in / 8); }

// Exposed so tests can pin the rounding helper against a library conversion.
uint16_t orc_bf16_round(float f) { return float_to_bf16_bits_rne(f); }

// [Math] + [Infra] compression: packed signs and alpha = mean|Δ| over the
// scope (whole matrix when per_row == 0, each output row when per_row == 1).
// alpha32 receives the float32 value the method stores; alpha64 (may be null)
// the fp64 mean before that rounding.
void orc_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in,
                  int per_row, uint8_t* packed, float* alpha32, double* alpha64) {
  const int64_t row_bytes = d_in / 8;
  CompensatedSum whole;
  for (int64_t r = 0; r < d_out; ++r) {
    // Sign bits, packed LSB first.
    for (int64_t k = 0; k < row_bytes; ++k) {
      unsigned byte = 0;
      for (int j = 0; j < 8; ++j) {
        const int64_t idx = r * d_in + 8 * k + j;
        byte |= static_cast<unsigned>(sign_bit(w_base, w_ft, idx)) << j;
      }
      packed[r * row_bytes + k] = static_cast<uint8_t>(byte);
    }
    // ‖Δ‖₁ over the row.
    CompensatedSum row_sum;
    for (int64_t c = 0; c < d_in; ++c) {
      const double a = std::fabs(delta_at(w_base, w_ft, r * d_in + c));
      row_sum.add(a);
      whole.add(a);
    }
    if (per_row) {
      const double mean = row_sum.value() / static_cast<double>(d_in);
      alpha32[r] = static_cast<float>(mean);
      if (alpha64) alpha64[r] = mean;
    }
  }
  if (!per_row) {
    const double mean = whole.value() / (static_cast<double>(d_out) * static_cast<double>(d_in));
    alpha32[0] = static_cast<float>(mean);
    if (alpha64) alpha64[0] = mean;
  }
}

// [Serving] step 3 of the request pipeline written to memory:
// W_eff = bf16(fp32(W_base) + α·(±1)).
void orc_reconstruct(const uint16_t* w_base, const uint8_t* packed, const float* alpha, int per_row,
                     int64_t d_out, int64_t d_in, uint16_t* w_eff) {
  for (int64_t r = 0; r < d_out; ++r) {
    const float a = alpha_for_row(alpha, per_row, r);
    for (int64_t c = 0; c < d_in; ++c) {
      const int64_t idx = r * d_in + c;
      w_eff[idx] = effective_weight(w_base[idx], packed_bit(packed, d_in, r, c), a);
    }
  }
}

// [Serving] conceptual fused_bitdelta_linear: y = x · W_effᵀ, fp64 sums.
// x is [M, d_in]; y is [M, d_out] in fp64.
void orc_linear(const uint16_t* x, int64_t M, const uint16_t* w_base, const uint8_t* packed,
                const float* alpha, int per_row, int64_t d_out, int64_t d_in, double* y) {
  double* w_row = new double[d_in > 0 ? d_in : 1];
  for (int64_t n = 0; n < d_out; ++n) {
    const float a = alpha_for_row(alpha, per_row, n);
    for (int64_t k = 0; k < d_in; ++k)
      w_row[k] = bf16_bits_to_float(
          effective_weight(w_base[n * d_in + k], packed_bit(packed, d_in, n, k), a));
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0;
      for (int64_t k = 0; k < d_in; ++k)
        acc += static_cast<double>(bf16_bits_to_float(x[m * d_in + k])) * w_row[k];
      y[m * d_out + n] = acc;
    }
  }
  delete[] w_row;
}

// [Math] the effective weight as the real number W_base + α·sign(Δ), before
// any rounding to a storage dtype: y = x·W_baseᵀ + α ⊙ (x·Sᵀ) with S = ±1 from
// the packed bits, every product and sum in fp64 (x·W_base products of two
// bf16 values and α·(±1) are exact in fp64).  The decode kernels compute this
// split form; it differs from orc_linear only by the bf16 rounding of W_eff.
void orc_linear_split(const uint16_t* x, int64_t M, const uint16_t* w_base,
                      const uint8_t* packed, const float* alpha, int per_row, int64_t d_out,
                      int64_t d_in, double* y) {
  for (int64_t n = 0; n < d_out; ++n) {
    const double a = static_cast<double>(alpha_for_row(alpha, per_row, n));
    for (int64_t m = 0; m < M; ++m) {
      double base = 0.0, signs = 0.0;
      for (int64_t k = 0; k < d_in; ++k) {
        const double xv = static_cast<double>(bf16_bits_to_float(x[m * d_in + k]));
        base += xv * static_cast<double>(bf16_bits_to_float(w_base[n * d_in + k]));
        signs += packed_bit(packed, d_in, n, k) ? xv : -xv;
      }
      y[m * d_out + n] = base + a * signs;
    }
  }
}

// The same linear, one output element at a time: y_out[i] = y[m_idx[i]][n_idx[i]].
void orc_linear_at(const uint16_t* x, int64_t M, const uint16_t* w_base, const uint8_t* packed,
                   const float* alpha, int per_row, int64_t d_out, int64_t d_in,
                   const int64_t* m_idx, const int64_t* n_idx, int64_t count, double* y_out) {
  (void)M;
  (void)d_out;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t m = m_idx[i];
    const int64_t n = n_idx[i];
    const float a = alpha_for_row(alpha, per_row, n);
    double acc = 0.0;
    for (int64_t k = 0; k < d_in; ++k) {
      const double w = bf16_bits_to_float(
          effective_weight(w_base[n * d_in + k], packed_bit(packed, d_in, n, k), a));
      acc += static_cast<double>(bf16_bits_to_float(x[m * d_in + k])) * w;
    }
    y_out[i] = acc;
  }
}

// [Serving] multi-tenant form: rows [seg_off[s], seg_off[s+1]) of x belong to a
// request for variant seg_var[s]; variant 0 is the base model (W_eff = W_base),
// variant v >= 1 uses packed[v-1] and alpha[v-1] over the shared W_base.
// One output element at a time, for the sampled (m, n) pairs.
void orc_linear_grouped_at(const uint16_t* x, int64_t M_total, const int32_t* seg_off,
                           const int32_t* seg_var, int32_t n_seg, const uint16_t* w_base,
                           const uint8_t* const* packed, const float* const* alpha, int32_t n_var,
                           int per_row, int64_t d_out, int64_t d_in, const int64_t* m_idx,
                           const int64_t* n_idx, int64_t count, double* y_out) {
  (void)M_total;
  (void)n_var;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t m = m_idx[i];
    const int64_t n = n_idx[i];
    int32_t seg = 0;
    while (seg < n_seg && !(seg_off[seg] <= m && m < seg_off[seg + 1])) ++seg;
    const int32_t v = seg_var[seg];
    double acc = 0.0;
    for (int64_t k = 0; k < d_in; ++k) {
      const uint16_t wb = w_base[n * d_in + k];
      double w;
      if (v == 0) {
        w = bf16_bits_to_float(wb);
      } else {
        const float a = alpha_for_row(alpha[v - 1], per_row, n);
        w = bf16_bits_to_float(effective_weight(wb, packed_bit(packed[v - 1], d_in, n, k), a));
      }
      acc += static_cast<double>(bf16_bits_to_float(x[m * d_in + k])) * w;
    }
    y_out[i] = acc;
  }
}

// Whole grouped output [M_total, d_out]: every segment through orc_linear with
// its variant (or the plain base product for variant 0).
void orc_linear_grouped(const uint16_t* x, int64_t M_total, const int32_t* seg_off,
                        const int32_t* seg_var, int32_t n_seg, const uint16_t* w_base,
                        const uint8_t* const* packed, const float* const* alpha, int32_t n_var,
                        int per_row, int64_t d_out, int64_t d_in, double* y) {
  (void)M_total;
  (void)n_var;
  for (int32_t s = 0; s < n_seg; ++s) {
    const int64_t m0 = seg_off[s];
    const int64_t rows = static_cast<int64_t>(seg_off[s + 1]) - m0;
    if (rows <= 0) continue;
    const int32_t v = seg_var[s];
    if (v == 0) {
      for (int64_t m = m0; m < m0 + rows; ++m)
        for (int64_t n = 0; n < d_out; ++n) {
          double acc = 0.0;
          for (int64_t k = 0; k < d_in; ++k)
            acc += static_cast<double>(bf16_bits_to_float(x[m * d_in + k])) *
                   static_cast<double>(bf16_bits_to_float(w_base[n * d_in + k]));
          y[m * d_out + n] = acc;
        }
    } else {
      orc_linear(x + m0 * d_in, rows, w_base, packed[v - 1], alpha[v - 1], per_row, d_out, d_in,
                 y + m0 * d_out);
    }
  }
}

// [K-Merge] Cosine similarity of two task vectors held in their 1-bit form:
// Δ̂ = α ⊙ S with S[n][k] = +1 / −1 from bit k of row n and α per row (or one
// α for the matrix).  cos = <Δ̂_a, Δ̂_b> / (‖Δ̂_a‖·‖Δ̂_b‖), every product and
// sum in fp64, element by element over the unpacked signs (the definition as
// written: no counting shortcut).  Outputs the three sums too.
void orc_sign_cosine(const uint8_t* packed_a, const float* alpha_a, const uint8_t* packed_b,
                     const float* alpha_b, int per_row, int64_t d_out, int64_t d_in,
                     double* out4) {
  const int64_t row_bytes = d_in / 8;
  double dot = 0.0, na = 0.0, nb = 0.0;
  for (int64_t r = 0; r < d_out; ++r) {
    const double a = static_cast<double>(alpha_for_row(alpha_a, per_row, r));
    const double b = static_cast<double>(alpha_for_row(alpha_b, per_row, r));
    for (int64_t c = 0; c < d_in; ++c) {
      const int bit_a = (packed_a[r * row_bytes + c / 8] >> (c % 8)) & 1;
      const int bit_b = (packed_b[r * row_bytes + c / 8] >> (c % 8)) & 1;
      const double ea = bit_a ? a : -a;
      const double eb = bit_b ? b : -b;
      dot += ea * eb;
      na += ea * ea;
      nb += eb * eb;
    }
  }
  out4[0] = dot / std::sqrt(na * nb);
  out4[1] = dot;
  out4[2] = na;
  out4[3] = nb;
}

}  // extern "C"
