// sp_oracle.cpp — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU definition of the per-token stage that the sequence-parallel
// rewrite places between ReduceScatter and AllGather:
//
//     AllReduce -> RMSNorm -> quant   ==>   ReduceScatter -> RMSNorm -> quant -> AllGather
//
// Sources (web pages; cited by title and section):
//   [SP/FC]    "vllm-ascend SP / FlashComm1 / FlashComm2" (ai6s.net), §2.1 core idea,
//              §2.2 mathematical equivalence, §2.3 code logic (the add-RMSNorm-bias pattern
//              and its ReduceScatter replacement), §2.4 limits (token padding to tp),
//              §3.3 code logic (pad -> reduce_scatter(dim 0) -> ... -> all_gather(dim 0) -> unpad).
//   [SP-Q]     "vLLM SP / AsyncTP / quantization tech notes" (beaiera.top), §四 "SP + AsyncTP
//              and quantization" (static FP8 / NVFP4 patterns, the per-tensor correctness table).
//   [PR18671]  "vllm-ascend PR #18671 解读: GLM V1 SP layout through DSA-CP", §2 (3500 tokens
//              padded to 3504, 16 contiguous 219-token shards), §5.2 (shard checks, zeroing of
//              padding rows), §5.3 (tail padding rows zeroed after the reduction).
//   [LongCat]  "基于Atlas A3集群的LongCat-Flash模型推理性能优化实践", o_proj TP paragraph
//              (reduce_scatter = element-wise sum, then split along the batch/token dim).
//
// This file shares no code, header, table or constant generator with the CUDA library. Only
// tests, the smoke check and the bench's CPU-baseline leg load it. Every computation below is
// written for a reader to check by eye: there is no blocking, fusion or reordering beyond the
// definition. Floating point is IEEE binary64 with the default round-to-nearest-even mode; the
// build passes -ffp-contract=off so that no multiply-add is fused on any host.
//
// Readings adopted where the pages are silent (each one is listed in the design notes):
//   * bias is added once after the reduction, before the norm: h = sum_r p_r + bias + residual
//     ([SP/FC] §2.3 passes a bias slot to the add-RMSNorm operator);
//   * a NULL residual is the "First" pattern of [SP-Q] §四 (no incoming residual);
//   * the norm and the quantiser act on the unrounded h and y (fused semantics);
//   * the static FP8 scale is a dequantisation scale: q = E4M3(y / scale);
//   * per-token FP8: s_t = max_j |y_j| / 448, stored as fp32; codes are relative to the stored
//     s_t; a row whose amax is 0 stores s_t = 0 and all-zero codes;
//   * NVFP4: gs is an encode multiplier; sf_b = E4M3(gs * amax_b / 6); codes
//     q = E2M1(y * gs / decode(sf_b)); element 2i in the low nibble of byte i; block scales
//     row-major [T_pad][H/16];
//   * where a floating-point value decides a code, the decision is taken on the fp32 rounding
//     of the quantiser input (the CUDA kernel's precision); everything before it is fp64;
//   * rows at or beyond T_valid are padding: their inputs are never read and every output byte
//     of those rows is zero ([PR18671] §5.2, §5.3).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// Status codes and quantisation modes: the numeric values of the library's C boundary,
// restated here so that both sides can be compared on invalid arguments.
enum Status { kOk = 0, kInvalidArg = 1, kUnsupported = 2, kAlignment = 3, kCuda = 4 };
enum Mode { kNone = 0, kFp8Static = 1, kFp8PerToken = 2, kNvfp4 = 3, kFp8DynamicPerTensor = 4 };

// ---------------------------------------------------------------------------------------------
// Number formats, from their published definitions (IEEE-style binary formats):
//   bfloat16  : 1 sign, 8 exponent (bias 127), 7 fraction bits; the top half of an IEEE binary32.
//   FP8 E4M3  : 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities; S.1111.111 is NaN,
//               so the largest finite magnitude is 1.75 * 2^8 = 448 (OCP 8-bit FP "E4M3").
//   FP4 E2M1  : 1 sign, 2 exponent (bias 1), 1 fraction bit; magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}
//               (OCP Microscaling formats).
// ---------------------------------------------------------------------------------------------
struct Format {
  int exp_bits;
  int frac_bits;
  int bias;
  double max_finite;
  bool saturate;  // true: clamp to +-max_finite ("satfinite"); false: overflow to infinity
};

const Format kBF16 = {8, 7, 127, std::ldexp(255.0, 120), false};  // (2 - 2^-7) * 2^127
const Format kE4M3 = {4, 3, 7, 448.0, true};
const Format kE2M1 = {2, 1, 1, 6.0, true};

// Nearest value of format f to x; ties go to the value with an even last fraction bit.
double round_to(double x, const Format& f) {
  if (x == 0.0 || std::isnan(x)) return x;
  const double a = std::fabs(x);
  if (std::isinf(a)) return f.saturate ? std::copysign(f.max_finite, x) : x;
  int e2 = 0;
  std::frexp(a, &e2);                                   // a = m * 2^e2, 0.5 <= m < 1
  const int emin = 1 - f.bias;                          // smallest normal exponent
  const int e = std::max(e2 - 1, emin);                 // binade of a (subnormals share emin's)
  const double quantum = std::ldexp(1.0, e - f.frac_bits);  // spacing of values in that binade
  const double n = std::nearbyint(a / quantum);         // exact scaling; rounds half to even
  double r = n * quantum;
  if (r > f.max_finite) r = f.saturate ? f.max_finite : INFINITY;
  return std::copysign(r, x);
}

// Bit pattern of a value that already lies on format f's grid (finite, not NaN).
unsigned encode_bits(double r, const Format& f) {
  const unsigned sign = std::signbit(r) ? 1u : 0u;
  const double a = std::fabs(r);
  unsigned field = 0, frac = 0;
  if (std::isinf(a)) {
    field = (1u << f.exp_bits) - 1u;
  } else if (a != 0.0) {
    int e2 = 0;
    std::frexp(a, &e2);
    const int e = e2 - 1;
    const int emin = 1 - f.bias;
    if (e < emin) {  // subnormal: a = frac * 2^(emin - frac_bits)
      field = 0;
      frac = static_cast<unsigned>(std::ldexp(a, f.frac_bits - emin));
    } else {         // normal: a = (1 + frac / 2^frac_bits) * 2^e
      field = static_cast<unsigned>(e + f.bias);
      frac = static_cast<unsigned>(std::ldexp(a / std::ldexp(1.0, e) - 1.0, f.frac_bits));
    }
  }
  return (sign << (f.exp_bits + f.frac_bits)) | (field << f.frac_bits) | frac;
}

// Value of a bit pattern of format f (E4M3's S.1111.111 is NaN; bf16's all-ones exponent is
// infinity or NaN as in binary32).
double decode_bits(unsigned code, const Format& f) {
  const unsigned frac_mask = (1u << f.frac_bits) - 1u;
  const unsigned exp_mask = (1u << f.exp_bits) - 1u;
  const unsigned frac = code & frac_mask;
  const unsigned field = (code >> f.frac_bits) & exp_mask;
  const bool neg = ((code >> (f.exp_bits + f.frac_bits)) & 1u) != 0;
  double mag;
  if (&f == &kE4M3 && field == exp_mask && frac == frac_mask) {
    mag = NAN;
  } else if (&f == &kBF16 && field == exp_mask) {
    mag = frac ? NAN : INFINITY;
  } else if (field == 0) {
    mag = std::ldexp(static_cast<double>(frac), 1 - f.bias - f.frac_bits);
  } else {
    mag = std::ldexp(1.0 + std::ldexp(static_cast<double>(frac), -f.frac_bits),
                     static_cast<int>(field) - f.bias);
  }
  return neg ? -mag : mag;
}

double bf16_value(uint16_t bits) { return decode_bits(bits, kBF16); }
uint16_t bf16_code(double x) { return static_cast<uint16_t>(encode_bits(round_to(x, kBF16), kBF16)); }
uint8_t e4m3_code(double x) { return static_cast<uint8_t>(encode_bits(round_to(x, kE4M3), kE4M3)); }
uint8_t e2m1_code(double x) { return static_cast<uint8_t>(encode_bits(round_to(x, kE2M1), kE2M1)); }

// The quantiser's decision is taken on the fp32 value of its input (see the file header).
double as_fp32(double v) { return static_cast<double>(static_cast<float>(v)); }

// ---------------------------------------------------------------------------------------------
// Argument rules. They restate the shard checks of [PR18671] §5.2 (padded token count equals
// local tokens * tp; the shard starts at rank * local tokens) in the form the single-GPU call
// sees them, plus the mode rules of [SP-Q] §四.
// ---------------------------------------------------------------------------------------------
struct Args {
  float partial_scale;        // multiplies every partial before the reduction (1 = none)
  const uint16_t* addend;     // bf16 [T_pad][H] added after the reduction, or null
  int scale_layout;           // NVFP4 block scales: 0 row-major, 1 128x4-tile swizzle
  const uint16_t* partials;
  int tp;
  int64_t T_pad;
  int64_t T_valid;
  int64_t H;
  const uint16_t* residual;
  const uint16_t* weight;
  const uint16_t* bias;
  float eps;
  int mode;
  const float* scale;
  void* out;
  void* out_scales;
  uint16_t* residual_out;
};

int64_t out_bytes(const Args& a) {
  switch (a.mode) {
    case kNone: return a.T_pad * a.H * 2;
    case kFp8Static:
    case kFp8PerToken: return a.T_pad * a.H;
    case kNvfp4: return a.T_pad * a.H / 2;
    default: return 0;
  }
}

// The 128x4-tile layout of NVFP4 block scales that block-scaled GEMMs read (cuBLAS "1D block
// scaling factors" layout): the [rows][cols] scale matrix is padded to multiples of 128 rows and
// 4 columns; tile (i, j) = rows 128i.., columns 4j.. is a 512-byte block at (i * tiles_per_row + j)
// * 512; inside it, row r and column c sit at (r % 32) * 16 + (r / 32) * 4 + c.
// Pinned on the CPU by PyTorch's own construction of this layout (a reshape/permute of the
// row-major scale matrix) and by the permutation property (every row-major scale once, padding
// zero); on the GPU cuBLASLt's block-scaled NVFP4 GEMM reads the library's output, whose parity
// with this function is tested.
int64_t swizzled_rows(int64_t T_pad) { return (T_pad + 127) / 128 * 128; }
int64_t swizzled_cols(int64_t H) { return (H / 16 + 3) / 4 * 4; }
int64_t swizzled_offset(int64_t row, int64_t col, int64_t H) {
  const int64_t tiles_per_row = swizzled_cols(H) / 4;
  const int64_t tile = (row / 128) * tiles_per_row + col / 4;
  const int64_t r = row % 128, c = col % 4;
  return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + c;
}

int64_t scale_bytes(const Args& a) {
  if (a.mode == kFp8PerToken) return a.T_pad * 4;
  if (a.mode == kNvfp4) {
    if (a.scale_layout == 1) return swizzled_rows(a.T_pad) * swizzled_cols(a.H);
    return a.T_pad * (a.H / 16);
  }
  return 0;
}

bool overlaps(const void* p, int64_t pn, const void* q, int64_t qn) {
  if (!p || !q || pn <= 0 || qn <= 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + static_cast<uintptr_t>(qn) && b < a + static_cast<uintptr_t>(pn);
}

int validate(const Args& a) {
  if (a.mode == kFp8DynamicPerTensor) return kUnsupported;  // not shard-local: [SP-Q] §四 table
  if (a.mode < kNone || a.mode > kNvfp4) return kInvalidArg;
  if (a.tp < 1 || a.T_pad < 0 || a.T_valid < 0 || a.T_valid > a.T_pad) return kInvalidArg;
  if (a.T_pad % a.tp != 0) return kInvalidArg;
  if (a.H <= 0 || a.H % 8 != 0) return kInvalidArg;
  if (a.mode == kNvfp4 && a.H % 16 != 0) return kInvalidArg;
  // The partials (the largest buffer, tp * T_pad * H bf16) stay below 2^62 bytes, so that every
  // byte count below fits in int64.
  if (a.T_pad > (int64_t{1} << 62) / (2 * a.H) / a.tp) return kInvalidArg;
  if (!(a.eps > 0.0f) || !std::isfinite(a.eps)) return kInvalidArg;
  if (a.T_pad == 0) return kOk;
  if (!a.partials || !a.weight || !a.out || !a.residual_out) return kInvalidArg;
  if ((a.mode == kFp8Static || a.mode == kNvfp4) && !a.scale) return kInvalidArg;
  if ((a.mode == kFp8PerToken || a.mode == kNvfp4) && !a.out_scales) return kInvalidArg;
  // Outputs must not overlap any input or each other; residual_out may be residual itself.
  const int64_t rows = a.T_pad * a.H * 2;
  if (!std::isfinite(a.partial_scale)) return kInvalidArg;
  if (a.scale_layout != 0 && a.scale_layout != 1) return kUnsupported;
  if (a.scale_layout == 1 && a.mode != kNvfp4) return kInvalidArg;
  const void* inputs[] = {a.partials, a.residual, a.weight, a.bias, a.scale, a.addend};
  const int64_t in_n[] = {rows * a.tp, rows, a.H * 2, a.H * 2, 4, rows};
  const void* outputs[] = {a.out, a.out_scales, a.residual_out};
  const int64_t out_n[] = {out_bytes(a), scale_bytes(a), rows};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 6; ++i) {
      if (o == 2 && i == 1 && a.residual_out == static_cast<const void*>(a.residual)) continue;
      if (overlaps(outputs[o], out_n[o], inputs[i], in_n[i])) return kInvalidArg;
    }
    for (int p = o + 1; p < 3; ++p)
      if (overlaps(outputs[o], out_n[o], outputs[p], out_n[p])) return kInvalidArg;
  }
  if (a.mode == kFp8Static || a.mode == kNvfp4) {
    const double s = *a.scale;
    if (!(s > 0.0) || !std::isfinite(s)) return kInvalidArg;
  }
  return kOk;
}

// ---------------------------------------------------------------------------------------------
// One token row t. Steps follow the rewritten pattern of [SP/FC] §2.3:
//   reduce_scatter(partials) -> add residual (and bias) -> RMSNorm(weight, eps) -> quant,
// with ReduceScatter's reduction being the element-wise sum over the tp partials ([LongCat],
// o_proj paragraph; [SP/FC] §3.3). On one device the scatter/gather are pure indexing: row t of
// the output is row t of the AllGather result ([SP/FC] §2.2 conclusion 1).
// ---------------------------------------------------------------------------------------------
// Where block scale (row t, block b) is stored.
uint8_t* scale_slot(const Args& a, int64_t t, int64_t b) {
  uint8_t* base = static_cast<uint8_t*>(a.out_scales);
  return a.scale_layout == 1 ? base + swizzled_offset(t, b, a.H) : base + t * (a.H / 16) + b;
}

void zero_row(const Args& a, int64_t t, double* y_out) {
  const int64_t H = a.H;
  std::memset(a.residual_out + t * H, 0, static_cast<size_t>(H) * 2);
  uint8_t* out = static_cast<uint8_t*>(a.out);
  switch (a.mode) {
    case kNone: std::memset(out + t * H * 2, 0, static_cast<size_t>(H) * 2); break;
    case kFp8Static: std::memset(out + t * H, 0, static_cast<size_t>(H)); break;
    case kFp8PerToken:
      std::memset(out + t * H, 0, static_cast<size_t>(H));
      static_cast<float*>(a.out_scales)[t] = 0.0f;
      break;
    case kNvfp4:
      std::memset(out + t * (H / 2), 0, static_cast<size_t>(H / 2));
      for (int64_t b = 0; b < H / 16; ++b) *scale_slot(a, t, b) = 0;
      break;
  }
  if (y_out) std::fill(y_out + t * H, y_out + (t + 1) * H, 0.0);
}

void one_row(const Args& a, int64_t t, double* y_out) {
  const int64_t H = a.H;
  if (t >= a.T_valid) {  // padding row: inputs never read, outputs all zero bytes
    zero_row(a, t, y_out);
    return;
  }
  std::vector<double> h(static_cast<size_t>(H)), y(static_cast<size_t>(H));

  // (1) reduction over the tp partial sums, r = 0 .. tp-1, each partial scaled first (a scale
  //     applied before the reduction: PR #18671 notes §5.3)
  // (2) h = reduced + bias + residual + addend (a missing term counts as zero; the addend is the
  //     per-shard extra input added between the ReduceScatter and the norm, SP/FlashComm notes
  //     §2.3, Qwen3-VL deepstack rewrite)
  const double ps = static_cast<double>(a.partial_scale);
  for (int64_t j = 0; j < H; ++j) {
    double s = 0.0;
    for (int r = 0; r < a.tp; ++r) s += ps * bf16_value(a.partials[(r * a.T_pad + t) * H + j]);
    const double b = a.bias ? bf16_value(a.bias[j]) : 0.0;
    const double res = a.residual ? bf16_value(a.residual[t * H + j]) : 0.0;
    const double add = a.addend ? bf16_value(a.addend[t * H + j]) : 0.0;
    h[j] = s + b + res + add;
  }

  // (3) the new residual is h rounded once to bf16 (read of row t above is complete, so
  //     residual_out may alias residual)
  for (int64_t j = 0; j < H; ++j) a.residual_out[t * H + j] = bf16_code(h[j]);

  // (4) RMSNorm over the hidden dimension of this one token: y = h / sqrt(mean(h^2) + eps) * w
  double sum_sq = 0.0;
  for (int64_t j = 0; j < H; ++j) sum_sq += h[j] * h[j];
  const double mean_sq = sum_sq / static_cast<double>(H);
  const double inv_rms = 1.0 / std::sqrt(mean_sq + static_cast<double>(a.eps));
  for (int64_t j = 0; j < H; ++j) y[j] = h[j] * inv_rms * bf16_value(a.weight[j]);
  if (y_out) std::copy(y.begin(), y.end(), y_out + t * H);

  // (5) output in the requested form
  uint8_t* out8 = static_cast<uint8_t*>(a.out);
  if (a.mode == kNone) {
    uint16_t* out16 = static_cast<uint16_t*>(a.out);
    for (int64_t j = 0; j < H; ++j) out16[t * H + j] = bf16_code(y[j]);
  } else if (a.mode == kFp8Static) {
    // static per-tensor: a calibrated constant, hence shard-local ([SP-Q] §四 table, row 1)
    const double scale = static_cast<double>(*a.scale);
    for (int64_t j = 0; j < H; ++j) out8[t * H + j] = e4m3_code(as_fp32(y[j] / scale));
  } else if (a.mode == kFp8PerToken) {
    // per-token: one scale per row, and a row belongs to one rank ([SP-Q] §四 table, row 3)
    double amax = 0.0;
    for (int64_t j = 0; j < H; ++j) amax = std::max(amax, std::fabs(y[j]));
    const float s_t = static_cast<float>(amax / 448.0);
    static_cast<float*>(a.out_scales)[t] = s_t;
    for (int64_t j = 0; j < H; ++j)
      out8[t * H + j] = (s_t == 0.0f) ? 0 : e4m3_code(as_fp32(y[j] / static_cast<double>(s_t)));
  } else if (a.mode == kNvfp4) {
    // per-block: 16-element blocks along H never cross a row, hence never a rank
    // ([SP-Q] §四 table, row 4)
    const double gs = static_cast<double>(*a.scale);
    uint8_t* q_row = out8 + t * (H / 2);
    for (int64_t b = 0; b < H / 16; ++b) {
      double amax = 0.0;
      for (int64_t j = 16 * b; j < 16 * b + 16; ++j) amax = std::max(amax, std::fabs(y[j]));
      const uint8_t sf = e4m3_code(as_fp32(gs * amax / 6.0));
      const double sf_value = decode_bits(sf, kE4M3);
      *scale_slot(a, t, b) = sf;
      for (int64_t j = 16 * b; j < 16 * b + 16; j += 2) {
        const uint8_t lo = sf_value == 0.0 ? 0 : e2m1_code(as_fp32(y[j] * gs / sf_value));
        const uint8_t hi = sf_value == 0.0 ? 0 : e2m1_code(as_fp32(y[j + 1] * gs / sf_value));
        q_row[j / 2] = static_cast<uint8_t>(lo | (hi << 4));
      }
    }
  }
}

Args make_args(const uint16_t* partials, int tp, int64_t T_pad, int64_t T_valid, int64_t H,
               const uint16_t* residual, const uint16_t* weight, const uint16_t* bias, float eps,
               int mode, const float* scale, void* out, void* out_scales, uint16_t* residual_out,
               float partial_scale = 1.0f, const uint16_t* addend = nullptr,
               int scale_layout = 0) {
  return Args{partial_scale, addend, scale_layout, partials, tp, T_pad, T_valid, H, residual,
              weight, bias, eps, mode, scale, out, out_scales, residual_out};
}

// Swizzled layout: every padding byte of the scale matrix (rows T_pad .. padded rows, columns
// H/16 .. padded columns) is zero.
void zero_scale_padding(const Args& a) {
  if (a.mode != kNvfp4 || a.scale_layout != 1) return;
  uint8_t* base = static_cast<uint8_t*>(a.out_scales);
  for (int64_t t = 0; t < swizzled_rows(a.T_pad); ++t)
    for (int64_t b = 0; b < swizzled_cols(a.H); ++b)
      if (t >= a.T_pad || b >= a.H / 16) base[swizzled_offset(t, b, a.H)] = 0;
}

}  // namespace

extern "C" {

// Whole call: rows 0 .. T_pad-1. Host pointers; same argument list and status codes as the
// library's device entry point (no stream).
int sp_oracle_fused_reduce_norm(const uint16_t* partials, int tp, int64_t T_pad, int64_t T_valid,
                                int64_t H, const uint16_t* residual, const uint16_t* weight,
                                const uint16_t* bias, float eps, int quant_mode, const float* scale,
                                void* out, void* out_scales, uint16_t* residual_out) {
  const Args a = make_args(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode,
                           scale, out, out_scales, residual_out);
  const int st = validate(a);
  if (st != kOk) return st;
  for (int64_t t = 0; t < T_pad; ++t) one_row(a, t, nullptr);
  return kOk;
}

// Rows [row_begin, row_end) only, and optionally the unrounded fp64 y of those rows into
// y_out[T_pad][H] (NULL to skip). Rows are independent, so disjoint ranges may run in parallel.
int sp_oracle_fused_reduce_norm_rows(const uint16_t* partials, int tp, int64_t T_pad,
                                     int64_t T_valid, int64_t H, const uint16_t* residual,
                                     const uint16_t* weight, const uint16_t* bias, float eps,
                                     int quant_mode, const float* scale, void* out,
                                     void* out_scales, uint16_t* residual_out, double* y_out,
                                     int64_t row_begin, int64_t row_end) {
  const Args a = make_args(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode,
                           scale, out, out_scales, residual_out);
  const int st = validate(a);
  if (st != kOk) return st;
  if (row_begin < 0 || row_end > T_pad || row_begin > row_end) return kInvalidArg;
  for (int64_t t = row_begin; t < row_end; ++t) one_row(a, t, y_out);
  return kOk;
}

// As sp_oracle_fused_reduce_norm_rows, with a scale applied to every partial before the
// reduction and an optional addend [T_pad][H] added after it (before the norm).
int sp_oracle_fused_reduce_norm_rows_ex(const uint16_t* partials, int tp, int64_t T_pad,
                                        int64_t T_valid, int64_t H, const uint16_t* residual,
                                        const uint16_t* weight, const uint16_t* bias, float eps,
                                        int quant_mode, const float* scale, void* out,
                                        void* out_scales, uint16_t* residual_out, double* y_out,
                                        int64_t row_begin, int64_t row_end, float partial_scale,
                                        const uint16_t* addend, int scale_layout) {
  const Args a = make_args(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode,
                           scale, out, out_scales, residual_out, partial_scale, addend,
                           scale_layout);
  const int st = validate(a);
  if (st != kOk) return st;
  if (row_begin < 0 || row_end > T_pad || row_begin > row_end) return kInvalidArg;
  if (row_begin == 0) zero_scale_padding(a);
  for (int64_t t = row_begin; t < row_end; ++t) one_row(a, t, y_out);
  return kOk;
}

// Size in bytes of out_scales for a mode and scale layout.
int64_t sp_oracle_out_scales_bytes(int64_t T_pad, int64_t H, int quant_mode, int scale_layout) {
  Args a{};
  a.T_pad = T_pad;
  a.H = H;
  a.mode = quant_mode;
  a.scale_layout = scale_layout;
  return scale_bytes(a);
}

// Argument rules alone.
int sp_oracle_check_args(const uint16_t* partials, int tp, int64_t T_pad, int64_t T_valid, int64_t H,
                         const uint16_t* residual, const uint16_t* weight, const uint16_t* bias,
                         float eps, int quant_mode, const float* scale, void* out,
                         void* out_scales, uint16_t* residual_out) {
  return validate(make_args(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                            quant_mode, scale, out, out_scales, residual_out));
}

// ---------------------------------------------------------------------------------------------
// FlashComm2 token reorganisation (SP/FlashComm notes §4.2-4.4, §4.7), all ranks on one host:
// x holds G = global_tp tensors [N][H/G] (rank r's feature slice of all N tokens, elements of
// `esize` bytes); y receives G tensors [N/D][H/P] (P = otp_size, D = odp_size = G/P).
// The steps as the page gives them:
//   ids   the reorganised batch ids: D lists, list j = token segments {j, j+D, j+2D, ...}
//         (P of the G segments of N/G tokens; [[0,2],[1,3]] for G=4, P=2);
//   (1)   every rank cuts its local tensor into D packets, packet j = the rows of list j's
//         segments, in list order;
//   (2)   all_to_all inside each ODP group {gD, ..., gD+D-1}: member j receives packet j of every
//         member m, in member order;
//   (3)   the received [D][rows][H/G] pieces are concatenated along the feature dimension.
// ---------------------------------------------------------------------------------------------
extern "C" void sp_oracle_fc2_batch_ids(int global_tp, int otp_size, int* ids /* [D][P] */) {
  const int D = global_tp / otp_size, P = otp_size;
  for (int j = 0; j < D; ++j)
    for (int k = 0; k < P; ++k) ids[j * P + k] = j + k * D;
}

extern "C" int sp_oracle_fc2_reorganize(const uint8_t* x, int global_tp, int otp_size, int64_t N,
                                        int64_t H, int esize, uint8_t* y) {
  const int G = global_tp;
  if (G < 1 || otp_size < 1 || G % otp_size != 0 || N % G != 0 || H % G != 0 || esize < 1)
    return kInvalidArg;
  const int P = otp_size, D = G / P;
  const int64_t seg = N / G, F = H / G, row_in = F * esize;
  std::vector<int> ids(static_cast<size_t>(D) * P);
  sp_oracle_fc2_batch_ids(G, P, ids.data());
  // (1) packets[s][j]: [P * seg][F]
  std::vector<std::vector<uint8_t>> packets(static_cast<size_t>(G) * D);
  for (int s = 0; s < G; ++s) {
    const uint8_t* local = x + static_cast<int64_t>(s) * N * row_in;
    for (int j = 0; j < D; ++j) {
      std::vector<uint8_t>& pk = packets[static_cast<size_t>(s) * D + j];
      for (int k = 0; k < P; ++k) {
        const int64_t first = ids[j * P + k] * seg;
        pk.insert(pk.end(), local + first * row_in, local + (first + seg) * row_in);
      }
    }
  }
  // (2) all_to_all in each ODP group, then (3) concat along features
  const int64_t rows_out = P * seg, row_out = static_cast<int64_t>(D) * row_in;
  for (int r = 0; r < G; ++r) {
    const int g = r / D, j = r % D;
    uint8_t* out = y + static_cast<int64_t>(r) * rows_out * row_out;
    for (int m = 0; m < D; ++m) {
      const std::vector<uint8_t>& recv = packets[static_cast<size_t>(g * D + m) * D + j];
      for (int64_t i = 0; i < rows_out; ++i)
        std::memcpy(out + i * row_out + m * row_in, recv.data() + i * row_in,
                    static_cast<size_t>(row_in));
    }
  }
  return kOk;
}

// Codecs, element-wise over n values (for the format tests).
void sp_oracle_bf16_encode(const double* x, uint16_t* code, int64_t n) {
  for (int64_t i = 0; i < n; ++i) code[i] = bf16_code(x[i]);
}
void sp_oracle_bf16_decode(const uint16_t* code, double* x, int64_t n) {
  for (int64_t i = 0; i < n; ++i) x[i] = bf16_value(code[i]);
}
void sp_oracle_e4m3_encode(const double* x, uint8_t* code, int64_t n) {
  for (int64_t i = 0; i < n; ++i) code[i] = e4m3_code(x[i]);
}
void sp_oracle_e4m3_decode(const uint8_t* code, double* x, int64_t n) {
  for (int64_t i = 0; i < n; ++i) x[i] = decode_bits(code[i], kE4M3);
}
void sp_oracle_e2m1_encode(const double* x, uint8_t* code, int64_t n) {
  for (int64_t i = 0; i < n; ++i) code[i] = e2m1_code(x[i]);
}
void sp_oracle_e2m1_decode(const uint8_t* code, double* x, int64_t n) {
  for (int64_t i = 0; i < n; ++i) x[i] = decode_bits(code[i] & 0xFu, kE2M1);
}

}  // extern "C"
