// Internal structures shared by the host side (psgd_api.cu) and the step
// kernels (psgd_kernels.cuh).  Plain structs copied to device memory once per
// context; nothing here allocates.
#pragma once

#include <stdint.h>

namespace psgd {

constexpr int kThreads = 64;      // threads per CTA of the step kernel (warps work alone)
constexpr int kWarps = kThreads / 32;
constexpr int kMaxWorkers = 64;   // W limit (pointer table passed by value)
constexpr int kSeg = 32;          // float4 columns per segment (one warp width)
constexpr int kGramGroup = 32;    // P1 row blocks whose Gram partials one group sums

// Work item kinds of the persistent step kernel, in dependency order.
enum ItemKind : int32_t {
  kItemP1 = 0,  // project: B_w <- G_w + E_w, P rows = sum_w M_w Q, Gram partial
  kItemPH = 1,  // orthonormalise: Phat rows = P rows R^-1 (needs the layer's Gram)
  kItemP3 = 2,  // back-project: partial Q_w = M_w^T Phat over a row tile (needs Phat)
  kItemU = 3,   // decompress: U rows = Phat Qbar^T (needs the layer's Qbar)
  kItemV = 4,   // vector layer: worker mean
};

struct Item {
  int32_t kind;
  int32_t layer;  // index into LayerDev (matrix) or VecDev (vector)
  int32_t a;      // row block (P1, U), item (PH, V) or row tile (P3)
  int32_t b;      // segment group (P1, U), segment * W + worker (P3), else 0
};

// One matrix layer: geometry, tiling and offsets into the context's buffers.
// Offsets are in elements of the respective buffer.  Every work item is
// processed by ONE warp.
struct LayerDev {
  int64_t off;       // offset in a packed gradient / B / U buffer
  int32_t n, m, ld;  // rows, columns, row stride (m rounded up to 4)
  int32_t F;         // float4 per row (ld / 4)
  int32_t S;         // segments of kSeg float4 per row
  int32_t tail;      // valid floats in the last float4 of a row (1..4)
  int32_t index;     // position of the layer in the caller's layer list
  // P1: items of r1 rows (sub-blocks of RS rows) x gs1 segments
  int32_t r1, nrb, gs1, nsg1;  // rows per item, row blocks, segments per item, segment groups
  int32_t g1;                  // Gram groups (kGramGroup row blocks each)
  // PH: items of 32 rows (one per lane)
  int32_t tph;
  // P3: items of r3 rows x one segment x one worker
  int32_t r3, t3r;
  // U: items of rsu rows x gsu segments
  int32_t rsu, gsu, nrbu, nsgu;
  int32_t pad0;
  int64_t p_off;      // P and Phat: n x RP
  int64_t q_off;      // Qbar: ld x RP; Q_w of worker w at w*q_total + q_off
  int64_t ppart_off;  // floats: nrb x nsg1 x r1 x RP partial P rows (nsg1 > 1)
  int64_t gram_off;   // doubles: (nrb + g1) x NG partial Grams
  int64_t rinv_off;   // doubles: RP x RP (R), RP (1 / diag R), RP x RP (Gram scratch)
  int64_t qpart_off;  // floats: t3r x W x ld x RP partial Q_w
  int32_t cnt_off;    // first counter of the layer; the others sit at cnt_off + c_*
  int32_t c_gram;     // Gram groups done (1)
  int32_t c_grp;      // row blocks done per Gram group (g1)
  int32_t c_ph;       // PH items done (1)
  int32_t c_qf;       // segments with Qbar done (1)
  int32_t c_qs;       // workers done per segment (S)
  int32_t c_p3;       // row tiles done per (segment, worker) (S x W)
  int32_t c_rb;       // P1 segment groups done per row block (nrb, when nsg1 > 1)
  int32_t flag_off;   // flags: [0] Gram ready, [1] Phat ready, [2] Qbar ready
  int32_t pad1;
};

struct VecDev {
  int64_t off;
  int32_t n;
  int32_t pad;
};

// Control block of one context (device memory, zeroed at create).
struct Ctl {
  unsigned next;      // work-queue head
  unsigned exited;    // warps that left the step kernel
  int status;         // 0, or a device-side error code (PSGD_ERR_TIMEOUT)
  int where;          // item index that recorded the error
};

constexpr int kDevTimeout = -4;  // equals PSGD_ERR_TIMEOUT

// One traced work item (optional, see psgd_options.trace): which item ran on
// which SM / warp slot, and its start and end on the global nanosecond timer.
struct TraceRec {
  uint32_t item;
  uint16_t sm;
  uint16_t warp;
  uint64_t t0, tw, t1;  // claimed, dependency wait over, done
};

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
  unsigned* flags;
  Ctl* ctl;
  const LayerDev* layers;
  const VecDev* vecs;
  const Item* items;
  int32_t num_items;
  int32_t W;
  unsigned epoch;               // step number (>= 1); flags hold the epoch that set them
  int32_t has_prev;             // 0 before the first step: no correction term
  int64_t spin_limit;
  TraceRec* trace;              // per-item timing records, or nullptr
};

}  // namespace psgd
