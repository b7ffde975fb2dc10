// Internal structures shared by the host side (psgd_api.cu) and the step
// kernels (psgd_kernels.cuh).  Plain structs copied to device memory once per
// context; nothing here allocates.
#pragma once

#include <stdint.h>

namespace psgd {

constexpr int kThreads = 256;     // threads per CTA of every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kMaxWorkers = 64;   // W limit (pointer table passed by value)
constexpr int kSeg = 32;          // float4 columns per segment (one warp width)
constexpr int kGramGroup = 32;    // P1 tiles whose Gram partials one group sums

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
  int32_t a;      // tile index (P1, PH, U, V) or row tile (P3)
  int32_t b;      // P3: segment * W + worker, else 0
};

// One matrix layer: geometry, tiling and offsets into the context's buffers.
// Offsets are in elements of the respective buffer.
struct LayerDev {
  int64_t off;       // offset in a packed gradient / B / U buffer
  int32_t n, m, ld;  // rows, columns, row stride (m rounded up to 4)
  int32_t F;         // float4 per row (ld / 4)
  int32_t S;         // segments of kSeg float4 per row
  int32_t tail;      // valid floats in the last float4 of a row (1..4)
  // P1: tiles of r1 rows, worked as (segment, sub-block) pairs of rs1 rows
  int32_t rs1, rho1, r1, t1;
  int32_t g1;        // Gram groups (kGramGroup tiles each)
  // PH: tiles of rph rows, one row per thread
  int32_t rph, tph;
  // P3: tiles of r3 rows x one segment x one worker (warps split the rows)
  int32_t r3, t3r;
  // U: like P1 with rsu rows per pair
  int32_t rsu, rhou, ru, tu;
  int32_t index;      // position of the layer in the caller's layer list
  int64_t p_off;      // P and Phat: n x RP
  int64_t q_off;      // Qbar: ld x RP; Q_w of worker w at w*q_total + q_off
  int64_t gram_off;   // doubles: (t1 + g1) x NG partial Grams
  int64_t rinv_off;   // doubles: RP x RP
  int64_t qpart_off;  // floats: t3r x W x ld x RP partial Q_w
  int32_t cnt_off;    // counters: [0] Gram groups done, [1..g1] tiles per Gram group,
                      // [1+g1] PH tiles, [2+g1] segments finalised, [3+g1+s] P3 tiles of segment s
  int32_t flag_off;   // flags: [0] Gram ready, [1] Phat ready, [2] Qbar ready
};

struct VecDev {
  int64_t off;
  int32_t n;
  int32_t pad;
};

// Control block of one context (device memory, zeroed at create).
struct Ctl {
  unsigned next;      // work-queue head
  unsigned exited;    // CTAs that left the step kernel
  int status;         // 0, or a device-side error code (PSGD_ERR_TIMEOUT)
  int where;          // item index that recorded the error
};

constexpr int kDevTimeout = -4;  // equals PSGD_ERR_TIMEOUT

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
};

}  // namespace psgd
