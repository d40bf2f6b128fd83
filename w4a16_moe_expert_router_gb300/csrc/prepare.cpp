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
// GEMM row r of block b is, for gate_up (R = 2f), gate row 64b+r for r < 64 and
// up row f+64b+r-64 for r >= 64 (so a block's tensor-memory lanes 0..63 hold
// gate rows and 64..127 the matching up rows); for down (R = d) it is row
// 128b+r.  The codes of a stage are ordered [half h][GEMM row r][4 words]:
// half h covers the stage's columns 32h .. 32h+31, and word w of (h, r) holds the
// 8 codes of row r at columns c0 = 32h + 8w + {0..7} (relative to the stage),
// nibble i (bits 4i..4i+3) holding column c0 + {0, 2, 4, 6, 1, 3, 5, 7}[i], the
// order in which the kernels' dequantiser produces the f16x2 column pairs
// (c0, c0+1), (c0+2, c0+3), ... it writes to tensor memory.  Each thread of the
// dequantiser reads its row's two 16-byte halves.
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
  if (p.gate_up) return r < 64 ? 64 * b + r : p.f + 64 * b + (r - 64);
  return moe::kBlockRows * b + r;
}

inline int groups_in_stage(int64_t s, int64_t g) {
  return g <= moe::kStageK ? int(moe::kStageK / g) : ((s * moe::kStageK) % g == 0 ? 1 : 0);
}

// Column offset (within a word's 8 columns) of nibble i of the word.
constexpr int kNibCol[8] = {0, 2, 4, 6, 1, 3, 5, 7};

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
        for (int hf = 0; hf < 2; ++hf) {
          for (int r = 0; r < moe::kBlockRows; ++r) {
            uint8_t* qrow = qe + rows[r] * rowb;
            for (int w = 0; w < 4; ++w) {
              const int64_t c0 = s * moe::kStageK + hf * 32 + w * 8;
              uint32_t word = 0;
              if (!kPack) std::memcpy(&word, out, 4);
              for (int i = 0; i < 8; ++i) {
                const int64_t col = c0 + kNibCol[i];
                uint8_t* byte = qrow + (col >> 1);
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
