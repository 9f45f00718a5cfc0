// Packed device layout of the expert weights (host and device code).
//
// Both formats are stored as 16-row tiles whose bytes are laid out in the
// order the tensor-core fragments of the expert kernels consume them, so every
// warp load is a 512-byte, 16-byte-per-lane coalesced vector (16-byte-aligned
// blocks: "Strata on an Intel Arc", alignment item of "Planned"; weights packed
// in the layout the tensor-core kernels read: knivesysl README).
//
// k-permutation.  An m16n8k16 step gives lane (g = lane/4, t = lane%4) the
// A-slots {2t, 2t+1, 2t+8, 2t+9} of rows g and g+8.  Within a 64-column chunk
// c, step w in 0..3 maps those slots to the original columns
//     64c + 16t + 4w + {0, 1, 2, 3}
// so each lane owns one whole 16-column block of its two rows per chunk (one
// NVFP4 scale per row, no replication).  The B operand (activations) uses the
// same map, so the product is unchanged.
//
// NVFP4 tile (K % 64 == 0, C = K/64 chunks, super-chunks of up to 8 chunks):
//   per super-chunk s: [scale vector 32 x 16 B][code vector j = 0..nc-1: 32 x 16 B]
//   scale vector, lane (g,t): byte 2j = e4m3 of (row g, block 4(8s+j)+t),
//                             byte 2j+1 = same block of row g+8.
//   code vector j, lane (g,t): word w = bytes [ (g, 4w..4w+1), (g+8, 4w..4w+1),
//                              (g, 4w+2..4w+3), (g+8, 4w+2..4w+3) ] of the lane's
//                              16-column block (low nibble = lower column).
// FP6 tile (K % 128 == 0, P = K/128 blocks = chunk pairs, super-chunks of up to 8 pairs):
//   per super-chunk s: [exponent vector 32 x 4 B][pair j: 3 vectors x 32 x 16 B]
//   exponent word, lane (g,t): bytes [E(g, 2t), E(g+8, 2t), E(g, 2t+1), E(g+8, 2t+1)]
//                              of the super-chunk's local blocks.
//   pair j, lane: 12 words; word h*6 + q*3 + {0,1,2} = {Ha, Hb, L} for chunk h
//   of the pair and step group q (steps 2q, 2q+1): Ha/Hb hold the high 4 bits
//   of 8 codes each, L the low 2 bits of 16 codes; unpacking gives the byte
//   containers U(w) = [(g,4w),(g,4w+1),(g+8,4w),(g+8,4w+1)] and
//   V(w) = [(g,4w+2),(g,4w+3),(g+8,4w+2),(g+8,4w+3)]:
//     U(2q) = (Ha<<2 & 0x3C..) | (L & 0x03..)      V(2q) = (Ha>>2 & 0x3C..) | (L>>2 & 0x03..)
//     U(2q+1) = (Hb<<2 & 0x3C..) | (L>>4 & 0x03..) V(2q+1) = (Hb>>2 & 0x3C..) | (L>>6 & 0x03..)
//   vector i of pair j sits at 128 + 1536 j + 512 i + 16 lane.
// Expert: [gate/up: I/16 tile pairs, each (gate tile, up tile)][down: H/16 tiles].
#pragma once

#include <stdint.h>

namespace moe {

enum { FMT_NVFP4 = 1, FMT_FP6 = 2 };

struct MatGeom {
  int K;        // reduction length
  int units;    // NVFP4: 64-column chunks; FP6: 128-column pairs
  int nsc;      // super-chunks per tile
  int sc_bytes; // bytes of a full super-chunk
  int tile_bytes;
};

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

MOE_HD MatGeom mat_geom(int fmt, int K) {
  MatGeom g;
  g.K = K;
  if (fmt == FMT_NVFP4) {
    g.units = K / 64;
    g.nsc = (g.units + 7) / 8;
    g.sc_bytes = 512 * 9;
    g.tile_bytes = 512 * (g.nsc + g.units);
  } else {
    g.units = K / 128;
    g.nsc = (g.units + 7) / 8;
    g.sc_bytes = 128 + 1536 * 8;
    g.tile_bytes = 128 * g.nsc + 1536 * g.units;
  }
  return g;
}

// units (chunks or pairs) in super-chunk s
MOE_HD int sc_units(const MatGeom& g, int s) {
  int n = g.units - 8 * s;
  return n < 8 ? n : 8;
}

struct ExpertGeom {
  MatGeom gu;       // gate / up: K = H
  MatGeom dn;       // down: K = I
  uint64_t gu_bytes;      // all gate/up tile pairs
  uint64_t expert_bytes;  // gate/up + down
};

MOE_HD ExpertGeom expert_geom(int fmt, int H, int I) {
  ExpertGeom e;
  e.gu = mat_geom(fmt, H);
  e.dn = mat_geom(fmt, I);
  e.gu_bytes = (uint64_t)(I / 16) * 2u * (uint64_t)e.gu.tile_bytes;
  e.expert_bytes = e.gu_bytes + (uint64_t)(H / 16) * (uint64_t)e.dn.tile_bytes;
  return e;
}

// Byte offset of 16-row tile `r` of matrix `m` (0 gate, 1 up, 2 down) within an expert.
MOE_HD uint64_t tile_offset(const ExpertGeom& e, int m, int r) {
  if (m == 2) return e.gu_bytes + (uint64_t)r * e.dn.tile_bytes;
  return ((uint64_t)r * 2u + (uint64_t)m) * (uint64_t)e.gu.tile_bytes;
}

// MMA layout of an NVFP4 matrix region (a second copy of the packed tiles,
// kept for the block-scaled tensor-core GEMMs): M rows in tile order (gate/up:
// M = 2I, 16-row gate and up tiles alternating; down: M = H), K columns, in
// stages of 256 columns (KS = ceil(K/256));
//   codes  [KS][M][128 B]: row r's columns 256s .. 256s + 255 in natural order
//          (low nibble = lower column, zero past K), so that the 128 rows x
//          128 bytes of a stage of an M-block are one contiguous 16 KB read;
//   scales [KS][M/128 blocks][4 K-steps of 64][512 B], a K-step's 512 bytes
//          holding row r's 4 block scales at (r % 32) * 16 + (r / 32) * 4 + b
//          (the groups tcgen05.cp moves).
// Per expert: gate/up codes, gate/up scales, down codes, down scales.
struct MmaGeom {
  int M, K, KS;
  uint64_t codes, scales;  // bytes
};

MOE_HD MmaGeom mma_geom(int M, int K) {
  MmaGeom g;
  g.M = M;
  g.K = K;
  g.KS = (K + 255) / 256;
  g.codes = (uint64_t)g.KS * (uint64_t)M * 128u;
  g.scales = (uint64_t)g.KS * (uint64_t)(M / 128) * 2048u;
  return g;
}

}  // namespace moe
