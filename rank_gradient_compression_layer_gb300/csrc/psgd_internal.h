// Internal structures shared by the host side (psgd_api.cu) and the phase
// kernels (psgd_kernels.cuh).  Plain structs copied to device memory once per
// context; nothing here allocates.
#pragma once

#include <stdint.h>

namespace psgd {

constexpr int kMaxWorkers = 64;   // W limit (pointer table passed by value)
constexpr int kSeg = 32;          // float4 columns per segment (one warp width)
constexpr int kGramGroup = 32;    // project row blocks whose Gram partials one group sums
// Share of L2 the error rows the back-project reads first may hold, stored
// by the project phase with an evict-last policy.
constexpr double kL2KeepShare = 0.3;
// Rows of one orthonormalise tile (one thread per row): fewer at large r, so
// that the tiles' float64 work (about r^2 per row) spreads over more SMs.
constexpr int ph_rows(int rp) { return rp >= 32 ? 32 : (rp == 16 ? 64 : 128); }
// Threads of an orthonormalise CTA: the row threads plus helpers for the
// second pass's partial-Gram sums (whose cost is load latency, not rows).
constexpr int kPhThreads = 128;
// Groups of kGramGroup orthonormalise tiles whose second-pass Gram partials
// one group sum takes.
constexpr int64_t ph_groups(int64_t nph) { return (nph + kGramGroup - 1) / kGramGroup; }
// Partial-Gram slots (NG doubles each) of a layer: project row blocks,
// project groups, orthonormalise tiles, orthonormalise groups.
constexpr int64_t gram_slots(int64_t nrb, int64_t g1, int64_t nph) { return nrb + g1 + nph + ph_groups(nph); }

// Doubles per layer of the factor record: R of the first Cholesky-QR pass
// (RP x RP, row-major) and 1 / diag R (RP); X = R2^-1 of the second pass
// (RP x RP, upper triangular) -- or, when the one-pass back-project applies,
// R^-1; a flag that is 1 when the first pass alone is orthogonal enough
// (then Phat = P1 and no second pass is formed); a flag that is 1 when the
// project phase formed Y_w = M_w^T P and P is well enough conditioned that
// Q_w = Y_w R^-1 (the back-project then reads no M).
constexpr int64_t rinv_len(int rp) { return 2 * (int64_t)rp * rp + rp + 2; }

// The one-pass project (padded rank <= 4): clusters of CTAs that together
// cover whole rows of a layer, so that a row block's P rows are complete on
// chip and Y_w = M_w^T P is accumulated in the same pass.
constexpr int kBmmaTmemCols = 512;  // tensor-core back-project: TMEM columns for every worker's D (W r)
constexpr int kYThreads = 256;     // threads of a CTA
constexpr int kYClusterMax = 8;    // CTAs per cluster (portable cluster size)
constexpr int kYSmemMax = 64 * 1024;  // Y accumulators of a CTA at most (bytes), so 3 CTAs fit on an SM
// M bytes a CTA writes per block at most (where a block of one row is not
// larger): the rows are read back two blocks later, and the whole GPU's
// blocks in between must stay in L2
constexpr int kYBlockBytes = 64 * 1024;
// kappa_F(R)^2 = ||R||_F^2 ||R^-1||_F^2 at most, for Q_w = Y_w R^-1: its
// rounding error is about kappa times that of Q_w = M_w^T Phat.
constexpr double kYKappa2 = 128.0 * 128.0;
__host__ __device__ constexpr int y_rows(int rp) { return 16 / rp; }       // rows of a block at most

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
  int64_t gram_off;   // doubles: gram_slots(nrb, g1, nph) x NG partial Grams (P, then P1)
  int64_t rinv_off;   // doubles: rinv_len(RP), the factor record
  int64_t qpart_off;  // floats: t3r x W x ld x RP partial Q_w
  int32_t cnt_off;    // first counter of the layer; the others sit at cnt_off + c_*
  int32_t c_gram;     // Gram groups done (1)
  int32_t c_grp;      // row blocks done per Gram group (g1)
  int32_t c_qs;       // workers done per segment (S)
  int32_t c_p3;       // row tiles done per (segment, worker) (S x W)
  int32_t c_rb;       // project column blocks done per row block (nrb, when s1 > 1)
  int32_t nph;        // orthonormalise tiles (rph rows each)
  int32_t c_ph;       // orthonormalise tiles (one pass) or tile groups (two passes) done (1)
  int32_t f_off;      // fused step: first of the layer's 2 + S flags (R ready, X ready, Qbar per segment)
  int32_t rph;        // rows per orthonormalise tile (ph_rows)
  int32_t s1;         // project tiles per row block (column blocks: segments, or half segments)
  int32_t c_phg;      // orthonormalise tiles done per tile group, second pass (ph_groups(nph))
  int32_t l2row;      // project: rows >= l2row store M to B with an L2 evict-last policy (the
                      // back-project reads them first, from L2); n: none
  // one-pass project (cw = 0: the layer is not on it): cw CTAs across a row,
  // yfc float4 columns each (a cluster holds kYClusterMax / cw such
  // subgroups); nys partial slots, one per segment of the schedule, each
  // with a Gram partial (nys + ceil(nys / kGramGroup) slots of NG doubles)
  // and a Y partial (W x ld x RP floats)
  int32_t cw, yfc, nys;
  int32_t c_yg;       // slots done per Gram group (ceil(nys / kGramGroup))
  int32_t yr;         // rows of a block (<= y_rows(RP)): a CTA's block of M stays about kYBlockBytes
  int64_t ygram_off;  // doubles
  int64_t y_off;      // floats
};

// The fused step runs every phase's tiles from one queue; an item is a Tile
// whose layer field carries the phase in its top byte.
enum ItemKind : int32_t { kItemProject = 0, kItemOrtho = 1, kItemBack = 2, kItemDecomp = 3 };
constexpr int32_t kLayerBits = 24;
constexpr int32_t item_layer(int32_t kind, int32_t layer) { return (kind << kLayerBits) | layer; }

// Flags of one matrix layer, relative to its f_off: each holds the number
// (epoch) of the last step that raised it.
constexpr int kFlagR = 0;     // R of the first Cholesky-QR pass stored
constexpr int kFlagX = 1;     // X = R2^-1 stored: the back-project may start
constexpr int kFlagQbar = 2;  // + segment: that segment's Qbar stored

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
  // fused step: the queue in `tiles` (n_items items, in dependency order),
  // the flags, and sync[0] = next ticket, sync[1] = CTAs finished,
  // sync[2] = status (0: ok, else the step was abandoned after a wait ran
  // past wait_ns); epoch = the value this step raises flags to
  unsigned* flags;
  unsigned* sync;
  int32_t n_items;
  uint32_t epoch;
  int64_t wait_ns;
  int32_t stall_layer;  // test hook: the R flag of this layer index is never raised (-1: none)
  // split step (workers spread over processes): the project phase stops
  // after writing this process's P (the sum over its workers; the Gram
  // factor follows once P has been all-reduced), and Qbar is
  // qbar_scale * sum over this process's workers of Q_w (1 / W in one process)
  int32_t split;
  float qbar_scale;
  // one-pass project: the project phase runs the cluster kernel, one
  // cluster per header tile (tiles[c] = {0, first segment, segments, 0}) over
  // segment tiles (tiles[y_clusters + i] = {layer, first block, end block,
  // first slot}), and writes Y partials here; the factor's last arriver
  // decides per layer whether the back-project uses them
  int32_t ypath;
  int32_t y_clusters;
  float* ypart;
};

}  // namespace psgd
