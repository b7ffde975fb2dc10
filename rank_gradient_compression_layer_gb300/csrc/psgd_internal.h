// Internal structures shared by the host side (psgd_api.cu) and the phase
// kernels (psgd_kernels.cuh).  Plain structs copied to device memory once per
// context; nothing here allocates.
#pragma once

#include <stdint.h>

namespace psgd {

constexpr int kMaxWorkers = 64;   // W limit (pointer table passed by value)
constexpr int kSeg = 32;          // float4 columns per segment (one warp width)
constexpr int kGramGroup = 32;    // project row blocks whose Gram partials one group sums

// One tile of a phase kernel (one CTA).  Meaning of the fields per phase:
//   project:        layer, row block, segment
//   orthonormalise: layer, row chunk
//   back-project:   layer, row tile, segment, worker
//   decompress:     layer, row block, segment, 0   |  vector layer, chunk, 0, 1
struct Tile {
  int32_t layer;
  int32_t a;
  int32_t b;
  int32_t c;
};

// One matrix layer: geometry, tiling and offsets into the context's buffers.
// Offsets are in elements of the respective buffer.
struct LayerDev {
  int64_t off;       // offset in a packed gradient / B / U buffer
  int32_t n, m, ld;  // rows, columns, row stride (m rounded up to 4)
  int32_t F;         // float4 per row (ld / 4)
  int32_t S;         // segments of kSeg float4 per row
  int32_t tail;      // valid floats in the last float4 of a row (1..4)
  int32_t index;     // position of the layer in the caller's layer list
  int32_t r1, nrb;   // project rows per tile (<= Cfg::R1), row blocks
  int32_t ru;        // decompress rows per tile (<= Cfg::RU)
  int32_t g1;        // Gram groups (kGramGroup row blocks each)
  int32_t r3, t3r;   // back-project rows per tile, row tiles
  int64_t p_off;      // P and Phat: n x RP (16-byte aligned)
  int64_t q_off;      // Qbar: ld x RP; Q_w of worker w at w*q_total + q_off
  int64_t ppart_off;  // floats: nrb x S x R1 x RP partial P rows (S > 1)
  int64_t gram_off;   // doubles: (nrb + g1) x NG partial Grams
  int64_t rinv_off;   // doubles: RP x RP (R), RP (1 / diag R)
  int64_t qpart_off;  // floats: t3r x W x ld x RP partial Q_w
  int32_t cnt_off;    // first counter of the layer; the others sit at cnt_off + c_*
  int32_t c_gram;     // Gram groups done (1)
  int32_t c_grp;      // row blocks done per Gram group (g1)
  int32_t c_qs;       // workers done per segment (S)
  int32_t c_p3;       // row tiles done per (segment, worker) (S x W)
  int32_t c_rb;       // segments done per row block (nrb, when S > 1)
};

struct VecDev {
  int64_t off;
  int32_t n;
  int32_t pad;
};

// Everything a phase kernel needs (passed by value).
struct StepArgs {
  const float* G[kMaxWorkers];  // per-worker packed gradients
  float* U;                     // packed update or nullptr
  float* B;                     // W x total: M of the last step (E = B - Phat Q_w^T)
  int64_t total;                // floats per packed buffer
  float* P;                     // sum over layers n x RP
  float* Phat;
  float* Qbar;                  // sum over layers ld x RP
  float* Qw;                    // W x q_total
  int64_t q_total;
  double* gram;
  double* rinv;
  float* qpart;
  float* ppart;
  unsigned* counters;
  const LayerDev* layers;
  const VecDev* vecs;
  const Tile* tiles;            // this phase's tiles
  int32_t W;
  int32_t has_prev;             // 0 before the first step: no correction term
  // optional momentum-SGD update fused into the decompress phase (packed
  // layout like U): Mom <- beta Mom + U, X <- X - lr (U + Mom); X == nullptr: off
  float* X;
  float* Mom;
  float lr;
  float beta;
  // unbiased variant: M = G (no error feedback, B untouched), P kept as is
  // (no Gram tail, no back-project), U = u_scale P Q^T with Q the step's draw
  int32_t unbiased;
  float u_scale;
};

}  // namespace psgd
