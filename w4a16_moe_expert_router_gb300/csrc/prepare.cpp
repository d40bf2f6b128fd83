// prepare.cpp -- host-side weight helpers: canonical nibble packing and the
// rearrangement into the stream the GEMM kernels consume.
//
// Canonical format (model card "srswti/axe-diffusion-ksl-xe", "requirements",
// dg-w4a16-v1): uint4 codes, two per byte along the contraction dim; this
// library reads byte b of a row as column 2b (low nibble) and column 2b+1 (high
// nibble); one fp16 scale and one fp16 zero-point per group of g columns.
//
// Prepared stream of one projection (rows R, contraction K, group g), per
// expert, per block of 128 GEMM rows, per stage of 128 columns (the last stage
// has 64 when K is an odd multiple of 64), per warp strip w = 0..7 of 16 GEMM rows:
//   [(scale, zero) pairs of the strip for the ng groups in this stage, 64 ng bytes]
//   [codes, 8 bytes per 16 columns per lane]
// GEMM row r of strip w of block b is, for gate_up (R = 2f), gate row
// 64b + 8w + r for r < 8 and up row f + 64b + 8w + r - 8 for r >= 8 (so one
// warp holds a gate row and its up row); for down (R = d) it is row
// 128b + 16w + r.  The (scale, zero) bytes are ordered [i = 0..7][group j]:
// 8 bytes holding the (scale, zero) of strip rows i and i + 8 for group j.  The
// codes are ordered [kk / 4][lane][kk % 4] (one 32-bit word per lane per 16-column
// step kk of the stage, so a lane reads four steps as one 16-byte vector and a
// warp's vector is 512 contiguous bytes); word (lane, kk) holds the lane's m16n8k16 A fragment of the 16 columns
// 16kk.. of the stage: with gq = lane / 4 and tq = lane % 4, nibble i (bits
// 4i..4i+3) is strip row gq + 8 (i & 1), column 16kk + 2tq + 8 ((i >> 1) & 1) + (i >> 2).
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <vector>

#include "internal.h"
#include "moe_w4a16.h"

namespace {

struct Proj {
  int64_t E, R, K, g, nblocks;
  bool gate_up;
  int64_t f;  // gate_up: the gate/up split
};

bool proj_of(const moe_w4a16_shape* sh, int32_t which, Proj* p) {
  if (!sh) return false;
  const size_t need = moe_w4a16_workspace_bytes(sh);
  if (need == 0) return false;  // invalid shape
  if (which == MOE_W4A16_GATE_UP) {
    *p = Proj{sh->experts, 2 * int64_t(sh->inter), sh->hidden, sh->group_gate_up, sh->inter / 64, true, sh->inter};
  } else if (which == MOE_W4A16_DOWN) {
    *p = Proj{sh->experts, sh->hidden, sh->inter, sh->group_down, sh->hidden / moe::kBlockRows, false, sh->inter};
  } else {
    return false;
  }
  return true;
}

constexpr int kStrips = moe::kBlockRows / moe::kStripRows;  // strips per block, one per compute warp
constexpr int64_t kStageCols = moe::kStageCols;

// Matrix row of row r (0..15) of strip w of block b.
inline int64_t strip_row(const Proj& p, int64_t b, int w, int r) {
  if (p.gate_up) return r < 8 ? 64 * b + 8 * w + r : p.f + 64 * b + 8 * w + (r - 8);
  return moe::kBlockRows * b + 16 * w + r;
}


double half_value(uint16_t h) {
  const int e = (h >> 10) & 31, m = h & 1023;
  double v = e == 0 ? std::ldexp(double(m), -24) : std::ldexp(1.0 + m / 1024.0, e - 15);
  if (e == 31) v = m ? NAN : INFINITY;
  return (h & 0x8000) ? -v : v;
}

template <bool kPack>
moe_w4a16_status walk(const Proj& p, uint8_t* q, uint16_t* scale, uint16_t* zero, uint8_t* stream) {
  const int64_t rowb = p.K / 2, ng = p.K / p.g;
  uint8_t* out = stream;
  for (int64_t e = 0; e < p.E; ++e) {
    uint8_t* qe = q + e * p.R * rowb;
    uint16_t* se = scale + e * p.R * ng;
    uint16_t* ze = zero + e * p.R * ng;
    for (int64_t b = 0; b < p.nblocks; ++b) {
      for (int64_t c0 = 0; c0 < p.K; c0 += kStageCols) {
        const int64_t width = std::min<int64_t>(kStageCols, p.K - c0);  // 128, or 64 for the last stage
        const int ngs = int(width / std::min<int64_t>(p.g, width));      // groups in the stage (g divides K)
        const int steps = int(width / 16);
        for (int w = 0; w < kStrips; ++w) {
          int64_t rows[16];
          for (int r = 0; r < 16; ++r) rows[r] = strip_row(p, b, w, r);
          for (int i = 0; i < 8; ++i) {
            for (int j = 0; j < ngs; ++j) {
              const int64_t grp = c0 / p.g + j;
              for (int h = 0; h < 2; ++h) {
                const int r = i + 8 * h;
                uint16_t* sp = se + rows[r] * ng + grp;
                uint16_t* zp = ze + rows[r] * ng + grp;
                if (kPack) {
                  std::memcpy(out, sp, 2);
                  std::memcpy(out + 2, zp, 2);
                } else {
                  std::memcpy(sp, out, 2);
                  std::memcpy(zp, out + 2, 2);
                }
                out += 4;
              }
            }
          }
          for (int kk = 0; kk < steps; ++kk) {
            for (int lane = 0; lane < 32; ++lane) {
              const int gq = lane >> 2, tq = lane & 3;
              uint8_t* wp = out + (kk / 4) * 512 + lane * 16 + (kk % 4) * 4;
              uint32_t word = 0;
              if (!kPack) std::memcpy(&word, wp, 4);
              for (int i = 0; i < 8; ++i) {
                const int r = gq + 8 * (i & 1);
                const int64_t col = c0 + 16 * kk + 2 * tq + 8 * ((i >> 1) & 1) + (i >> 2);
                uint8_t* byte = qe + rows[r] * rowb + (col >> 1);
                const int sh = (col & 1) ? 4 : 0;
                if (kPack) {
                  word |= uint32_t((*byte >> sh) & 15u) << (4 * i);
                } else {
                  const uint8_t code = uint8_t((word >> (4 * i)) & 15u);
                  *byte = uint8_t((*byte & ~(15u << sh)) | (code << sh));
                }
              }
              if (kPack) std::memcpy(wp, &word, 4);
            }
          }
          out += steps * 128;
        }
      }
    }
  }
  return MOE_W4A16_OK;
}

}  // namespace

extern "C" {

moe_w4a16_status moe_w4a16_pack(const uint8_t* codes, int64_t rows, int64_t K, uint8_t* packed) {
  if (!codes || !packed) return MOE_W4A16_ERR_NULL;
  if (rows < 0 || K < 0 || K % 2 != 0) return MOE_W4A16_ERR_SHAPE;
  for (int64_t i = 0; i < rows * K; ++i)
    if (codes[i] > 15) return MOE_W4A16_ERR_VALUE;
  for (int64_t i = 0; i < rows * K / 2; ++i) packed[i] = uint8_t(codes[2 * i] | (codes[2 * i + 1] << 4));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_unpack(const uint8_t* packed, int64_t rows, int64_t K, uint8_t* codes) {
  if (!codes || !packed) return MOE_W4A16_ERR_NULL;
  if (rows < 0 || K < 0 || K % 2 != 0) return MOE_W4A16_ERR_SHAPE;
  for (int64_t i = 0; i < rows * K / 2; ++i) {
    codes[2 * i] = packed[i] & 15u;
    codes[2 * i + 1] = packed[i] >> 4;
  }
  return MOE_W4A16_OK;
}

size_t moe_w4a16_prepared_bytes(const moe_w4a16_shape* shape, int32_t which) {
  Proj p;
  if (!proj_of(shape, which, &p)) return 0;
  return size_t(p.E * p.R * (p.K / 2) + p.E * p.R * (p.K / p.g) * 4);
}

moe_w4a16_status moe_w4a16_prepare(const moe_w4a16_shape* shape, int32_t which, const uint8_t* q,
                                   const uint16_t* scale, const uint16_t* zero, uint8_t* out) {
  if (!shape) return MOE_W4A16_ERR_NULL;
  Proj p;
  if (!proj_of(shape, which, &p)) return MOE_W4A16_ERR_SHAPE;
  const int fmt = shape->format;
  if (!q || !scale || !out || (!zero && fmt != 2)) return MOE_W4A16_ERR_NULL;
  const int64_t nsz = p.E * p.R * (p.K / p.g);
  std::vector<uint16_t> eights;
  if (fmt == 2) {  // symmetric: the zero-point slot holds 8 (0x4800), whatever zero points to
    eights.assign(size_t(nsz), uint16_t(0x4800));
    zero = eights.data();
  }
  for (int64_t i = 0; i < nsz; ++i) {
    const double s = half_value(scale[i]), z = half_value(zero[i]);
    if (!std::isfinite(s) || std::fabs(s) > 32.0) return MOE_W4A16_ERR_VALUE;
    if (fmt == 1 ? !(std::fabs(z) <= 1024.0) : !(z >= 0.0 && z <= 16.0)) return MOE_W4A16_ERR_VALUE;
  }
  return walk<true>(p, const_cast<uint8_t*>(q), const_cast<uint16_t*>(scale), const_cast<uint16_t*>(zero), out);
}

moe_w4a16_status moe_w4a16_unprepare(const moe_w4a16_shape* shape, int32_t which, const uint8_t* prepared,
                                     uint8_t* q, uint16_t* scale, uint16_t* zero) {
  if (!shape) return MOE_W4A16_ERR_NULL;
  Proj p;
  if (!proj_of(shape, which, &p)) return MOE_W4A16_ERR_SHAPE;
  if (!prepared || !q || !scale || (!zero && shape->format != 2)) return MOE_W4A16_ERR_NULL;
  std::memset(q, 0, size_t(p.E * p.R * (p.K / 2)));
  std::vector<uint16_t> scratch;
  if (!zero) {  // symmetric format without a zero-point array
    scratch.resize(size_t(p.E * p.R * (p.K / p.g)));
    zero = scratch.data();
  }
  return walk<false>(p, q, scale, zero, const_cast<uint8_t*>(prepared));
}

}  // extern "C"
