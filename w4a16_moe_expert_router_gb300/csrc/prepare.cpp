// prepare.cpp -- host-side weight helpers: canonical nibble packing and the
// rearrangement into the stream the GEMM kernels consume.
//
// Canonical format (model card "srswti/axe-diffusion-ksl-xe", "requirements",
// dg-w4a16-v1): uint4 codes, two per byte along the contraction dim; this
// library reads byte b of a row as column 2b (low nibble) and column 2b+1 (high
// nibble); one fp16 scale and one fp16 zero-point per group of g columns.
//
// Prepared stream of one projection (rows R, contraction K, group g), per
// expert, per block of 128 GEMM rows, per stage of 64 columns:
//   [(scale, zero) pairs of the block's 128 rows for each group starting in
//    this stage, 512 bytes per group][4096 bytes of codes]
// GEMM row order inside a block: 8 tiles of 16 rows.  For gate_up (R = 2f) tile
// m of block b holds gate rows 64b+8m .. +7 then up rows f+64b+8m .. +7; for down
// (R = d) it holds rows 128b+16m .. +15.  The codes of a stage are ordered
// [tile m][lane][k16 step], one 32-bit word each, a word holding the eight
// codes lane (g = lane/4, t = lane%4) needs for one m16n8k16 A fragment:
//   bits  0..3  (row g,   col 2t)    bits 16..19 (row g,   col 2t+1)
//   bits  4..7  (row g+8, col 2t)    bits 20..23 (row g+8, col 2t+1)
//   bits  8..11 (row g,   col 2t+8)  bits 24..27 (row g,   col 2t+9)
//   bits 12..15 (row g+8, col 2t+8)  bits 28..31 (row g+8, col 2t+9)
// (rows relative to the tile, columns relative to the k16 step).
#include <cmath>
#include <cstdint>
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

// Matrix row of GEMM row r (0..127) of block b.
inline int64_t gemm_row(const Proj& p, int64_t b, int r) {
  const int m = r >> 4, i = r & 15;
  if (p.gate_up) return i < 8 ? 64 * b + 8 * m + i : p.f + 64 * b + 8 * m + (i - 8);
  return moe::kBlockRows * b + r;
}

inline int groups_in_stage(int64_t s, int64_t g) {
  return g <= moe::kStageK ? int(moe::kStageK / g) : ((s * moe::kStageK) % g == 0 ? 1 : 0);
}

// Column offsets (within a k16 step) of nibble i of a word, and whether it is row g+8.
constexpr int kNibCol[8] = {0, 0, 8, 8, 1, 1, 9, 9};
constexpr int kNibHi[8] = {0, 1, 0, 1, 0, 1, 0, 1};

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
      int64_t rows[moe::kBlockRows];
      for (int r = 0; r < moe::kBlockRows; ++r) rows[r] = gemm_row(p, b, r);
      for (int64_t s = 0; s < p.K / moe::kStageK; ++s) {
        const int ngs = groups_in_stage(s, p.g);
        for (int j = 0; j < ngs; ++j) {
          const int64_t grp = (s * moe::kStageK) / p.g + j;
          for (int r = 0; r < moe::kBlockRows; ++r) {
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
        for (int m = 0; m < 8; ++m) {
          for (int lane = 0; lane < 32; ++lane) {
            const int gg = lane >> 2, t = lane & 3;
            for (int kk = 0; kk < 4; ++kk) {
              const int64_t c0 = s * moe::kStageK + kk * 16 + 2 * t;
              uint32_t word = 0;
              if (!kPack) std::memcpy(&word, out, 4);
              for (int i = 0; i < 8; ++i) {
                const int64_t row = rows[16 * m + gg + 8 * kNibHi[i]];
                const int64_t col = c0 + kNibCol[i];
                uint8_t* byte = qe + row * rowb + (col >> 1);
                const int sh = (col & 1) ? 4 : 0;
                if (kPack) {
                  word |= uint32_t((*byte >> sh) & 15u) << (4 * i);
                } else {
                  const uint8_t code = uint8_t((word >> (4 * i)) & 15u);
                  *byte = uint8_t((*byte & ~(15u << sh)) | (code << sh));
                }
              }
              if (kPack) std::memcpy(out, &word, 4);
              out += 4;
            }
          }
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
  if (!q || !scale || !zero || !out) return MOE_W4A16_ERR_NULL;
  const int64_t nsz = p.E * p.R * (p.K / p.g);
  for (int64_t i = 0; i < nsz; ++i) {
    const double s = half_value(scale[i]), z = half_value(zero[i]);
    if (!std::isfinite(s) || std::fabs(s) > 32.0) return MOE_W4A16_ERR_VALUE;
    if (!(z >= 0.0 && z <= 16.0)) return MOE_W4A16_ERR_VALUE;
  }
  return walk<true>(p, const_cast<uint8_t*>(q), const_cast<uint16_t*>(scale), const_cast<uint16_t*>(zero), out);
}

moe_w4a16_status moe_w4a16_unprepare(const moe_w4a16_shape* shape, int32_t which, const uint8_t* prepared,
                                     uint8_t* q, uint16_t* scale, uint16_t* zero) {
  if (!shape) return MOE_W4A16_ERR_NULL;
  Proj p;
  if (!proj_of(shape, which, &p)) return MOE_W4A16_ERR_SHAPE;
  if (!prepared || !q || !scale || !zero) return MOE_W4A16_ERR_NULL;
  std::memset(q, 0, size_t(p.E * p.R * (p.K / 2)));
  return walk<false>(p, q, scale, zero, const_cast<uint8_t*>(prepared));
}

}  // extern "C"
