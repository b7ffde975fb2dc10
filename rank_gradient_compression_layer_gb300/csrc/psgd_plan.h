// Host-side planning shared by the entry points of libpsgd.so: kernel set per
// padded rank, tile sizes of one matrix layer, the occupancy-driven choice of
// tile rows, and the error reporting behind psgd_last_error().
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "../../include/psgd.h"
#include "psgd_dispatch.h"

namespace psgd {

// Sets the calling thread's psgd_last_error() message and returns `code`.
int fail(int code, const char* fmt, ...);
// fail() with PSGD_ERR_OOM for an allocation failure, else PSGD_ERR_CUDA.
int cuda_fail(cudaError_t e, const char* what);

#define CUDA_TRY(x)                                  \
  do {                                               \
    cudaError_t e_ = (x);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #x); \
  } while (0)

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int padded_rank(int r) {
  int rp = 1;
  while (rp < r) rp *= 2;
  return rp;
}

inline const KernelSet* kernels_for(int rp) {
  switch (rp) {
    case 1: return &kKernelsR1;
    case 2: return &kKernelsR2;
    case 4: return &kKernelsR4;
    case 8: return &kKernelsR8;
    case 16: return &kKernelsR16;
    case 32: return &kKernelsR32;
    default: return nullptr;
  }
}

// Rows per tile of the project, back-project (least) and decompress phases.
// Whether the back-project runs on the tensor cores: padded rank 32 (at 16
// the CUDA-core kernel is faster: the tensor-core tile is bound by its shared
// memory traffic, hi and lo copies of M written and read three times), and
// every worker's D fits in TMEM.
inline bool bmma_applies(const KernelSet& ks, int W) {
  return ks.launch_bmma != nullptr && ks.rp == 32 && W * ks.rp <= kBmmaTmemCols;
}

struct TileRows {
  int r1 = 32, r3min = 512, ru = 64;
  int pcols = kSeg * 4;  // columns of a project tile
  int r3mult = 1;        // back-project rows per tile: a multiple of this (tensor-core chunks)
};

// The phase grids must hold several waves of resident CTAs, or the last,
// partly filled wave leaves HBM idle.  The back-project needs fewer: its
// tiles end in a cross-warp sum and a count, whose barriers cost more than
// the tail of fewer, taller tiles (one wave of 512-row tiles measured faster
// than two, four or eight waves on the ResNet-18 set).
constexpr int kWaves = 4;
constexpr int kBackWaves = 1;

// Tiling of one matrix layer for padded rank rp and W workers.  Returns the
// number of counters the layer needs and sets its counter offsets relative
// to cnt_off.
inline int64_t plan_matrix(LayerDev& L, int64_t n, int64_t m, int64_t ld, int rp, int W, const TileRows& tr) {
  L.n = (int32_t)n;
  L.m = (int32_t)m;
  L.ld = (int32_t)ld;
  L.F = (int32_t)(ld / 4);
  L.S = (int32_t)ceil_div(L.F, kSeg);
  L.tail = (int32_t)(m - 4 * (L.F - 1));
  L.r1 = tr.r1;
  L.nrb = (int32_t)ceil_div(n, L.r1);
  L.ru = tr.ru;
  L.g1 = (int32_t)ceil_div(L.nrb, kGramGroup);
  // back-project: at most 16 row tiles (the Q partial sums stay short)
  const int64_t r3 = ceil_div(std::max<int64_t>(std::max(tr.r3min, 8 * rp), ceil_div(n, 16)), tr.r3mult) * tr.r3mult;
  L.r3 = (int32_t)std::min<int64_t>(n, r3);
  L.t3r = (int32_t)ceil_div(n, L.r3);
  L.c_gram = 0;
  L.c_grp = 1;
  L.c_qs = 1 + L.g1;
  L.c_p3 = L.c_qs + L.S;
  L.c_rb = L.c_p3 + L.S * W;
  L.rph = ph_rows(rp);
  L.nph = (int32_t)ceil_div(n, L.rph);
  L.s1 = (int32_t)ceil_div(ld, tr.pcols);
  L.c_ph = L.c_rb + (L.s1 > 1 ? L.nrb : 0);
  L.c_phg = L.c_ph + 1;
  L.l2row = (int32_t)n;
  return (int64_t)L.c_phg + ph_groups(L.nph);
}

// Shared memory of a CTA's Y accumulators for `pairs` (float4 column,
// worker) pairs: RP float4 per pair, in whole rounds of kYThreads pairs.
inline int64_t y_smem_bytes(int64_t pairs, int rp) { return ceil_div(pairs, kYThreads) * kYThreads * rp * 16; }

// One-pass project, columns of a layer: cw CTAs across a row (1, 2, 4 or 8).
// A row's work is cw x ceil(pairs / kYThreads) rounds of (float4 column,
// worker) pairs per thread, pairs = ceil(F / cw) x W; cw is the one with the
// fewest rounds whose Y accumulators fit in kYSmemMax, ties going to the
// larger cw (fewer Y partials).  False when none fits.
inline bool plan_ycols(LayerDev& L, int rp, int W) {
  int best = 0;
  int64_t best_cost = 0;
  for (int cw = kYClusterMax; cw >= 1; cw /= 2) {
    const int64_t ps = ceil_div(L.F, cw) * W;
    if (y_smem_bytes(ps, rp) > kYSmemMax) continue;
    const int64_t cost = cw * ceil_div(ps, kYThreads);
    if (!best || cost < best_cost) {
      best = cw;
      best_cost = cost;
    }
  }
  if (!best) return false;
  L.cw = best;
  L.yfc = (int32_t)ceil_div(L.F, best);
  // rows of a block: at most y_rows(rp) and kYBlockBytes of M per CTA; then
  // as few as fill the same number of rounds of S blocks, so that the
  // layer's last round has no idle subgroups where it can be avoided
  const int64_t row_bytes = (int64_t)L.yfc * W * 16;
  const int64_t yr_max = std::min<int64_t>(y_rows(rp), std::max<int64_t>(1, kYBlockBytes / row_bytes));
  const int64_t S = kYClusterMax / best;
  const int64_t rounds = ceil_div(ceil_div((int64_t)L.n, yr_max), S);
  L.yr = (int32_t)ceil_div((int64_t)L.n, rounds * S);
  return true;
}

// A block of yr rows in units of a cluster's time: kYClusterMax / cw blocks
// run at once, each yr x ceil(pairs / kYThreads) rows of pair rounds long.
inline int64_t y_block_cost(const LayerDev& L, int W) {
  return (int64_t)L.cw * L.yr * ceil_div((int64_t)L.yfc * W, kYThreads);
}

// The one-pass project's persistent schedule for nc clusters: the layers'
// blocks of yr rows, in layer order, cut into nc runs of about equal cost;
// a run is a list of segments (layer, first block, end block, first slot),
// cut after the whole number of rounds (S = kYClusterMax / cw blocks, one per
// subgroup) nearest to each cluster's cumulative share of the total.
// Subgroup s of a segment takes its blocks
// s, s + S, ...; the segment's Y and Gram partials go to slot `first` (one
// per segment).  tiles = nc header tiles {0, first segment, segments, 0}
// followed by the segments.  Sets each layer's nys.
inline void plan_yschedule(std::vector<LayerDev>& hl, int rp, int W, int nc, std::vector<Tile>& tiles) {
  (void)rp;
  // a segment of k blocks takes ceil(k / S) rounds of one block's cost
  auto seg_cost = [&](const LayerDev& L, int64_t k) {
    const int64_t S = kYClusterMax / L.cw;
    return ceil_div(k, S) * S * y_block_cost(L, W);
  };
  int64_t total = 0;
  for (const LayerDev& L : hl) total += seg_cost(L, ceil_div(L.n, L.yr));
  std::vector<std::vector<Tile>> runs((size_t)nc);
  int c = 0;
  int64_t acc = 0;
  for (int li = 0; li < (int)hl.size(); ++li) {
    LayerDev& L = hl[li];
    L.nys = 0;
    const int64_t S = kYClusterMax / L.cw;
    const int64_t nb = ceil_div(L.n, L.yr), rc = S * y_block_cost(L, W);
    int64_t b = 0;
    while (b < nb) {
      int64_t k = nb - b;
      if (c + 1 < nc) {
        const int64_t room = total * (c + 1) / nc - acc;
        const int64_t kr = room > 0 ? (room + rc / 2) / rc : 0;  // the nearest whole number of rounds
        if (kr == 0) {
          ++c;
          continue;
        }
        k = std::min(k, kr * S);
      }
      runs[(size_t)c].push_back({li, (int32_t)b, (int32_t)(b + k), L.nys});
      L.nys += 1;
      acc += seg_cost(L, k);
      b += k;
    }
  }
  tiles.clear();
  int32_t first = 0;
  for (int i = 0; i < nc; ++i) {
    tiles.push_back({0, first, (int32_t)runs[(size_t)i].size(), 0});
    first += (int32_t)runs[(size_t)i].size();
  }
  for (const auto& r : runs) tiles.insert(tiles.end(), r.begin(), r.end());
}

// Chooses the tile rows of a layer set so that the project grid is at least
// kWaves waves of resident CTAs and the back-project grid kBackWaves (or the
// rows reach their floor); decompress tiles keep their size (their cost is
// the per-tile set-up, not the tail).
inline int choose_tile_rows(const std::vector<int64_t>& n, const std::vector<int64_t>& m, int rp, int W,
                            const KernelSet& ks, int device, TileRows* tr) {
  int sms = 0, c1 = 0, c3 = 0, cu = 0;
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
  CUDA_TRY(ks.occupancy(kProject, W, &c1));
  CUDA_TRY(ks.occupancy(kBackProject, W, &c3));
  CUDA_TRY(ks.occupancy(kDecompress, W, &cu));
  auto count = [&](int r1, int r3min, int ru, int64_t* t1, int64_t* t3, int64_t* tu) {
    *t1 = *t3 = *tu = 0;
    for (size_t l = 0; l < n.size(); ++l) {
      if (m[l] == 0) continue;
      const int64_t S = ceil_div(ceil_div(m[l], 4), kSeg);
      const int64_t r3 = std::min<int64_t>(n[l], std::max<int64_t>(std::max(r3min, 8 * rp), ceil_div(n[l], 16)));
      *t1 += ceil_div(n[l], r1) * S;
      *t3 += ceil_div(n[l], r3) * S * W;
      *tu += ceil_div(n[l], ru) * S;
    }
  };
  int64_t t1, t3, tu;
  TileRows r;
  r.r1 = ks.r1;
  r.ru = ks.ru;
  count(r.r1, r.r3min, r.ru, &t1, &t3, &tu);
  while (t1 < (int64_t)kWaves * c1 * sms && r.r1 > ks.rsb) {
    r.r1 /= 2;
    count(r.r1, r.r3min, r.ru, &t1, &t3, &tu);
  }
  while (t3 < (int64_t)kBackWaves * c3 * sms && r.r3min > 32) {
    r.r3min /= 2;
    count(r.r1, r.r3min, r.ru, &t1, &t3, &tu);
  }
  *tr = r;
  return PSGD_OK;
}

// The tiles of one matrix layer, per phase, in the order the phase kernels
// take them.  Back-project tiles run from the last row tile and segment to
// the first, so that they start on the rows the project tiles wrote last.
inline void layer_tiles(const LayerDev& L, int li, int W, std::vector<Tile> (&out)[kPhases]) {
  for (auto& v : out) v.clear();
  for (int rb = 0; rb < L.nrb; ++rb)
    for (int s = 0; s < L.s1; ++s) out[kProject].push_back({li, rb, s, 0});
  for (int t = 0; t < L.nph; ++t) out[kOrthonormalise].push_back({li, t, 0, 0});
  for (int rt = L.t3r - 1; rt >= 0; --rt)
    for (int s = L.S - 1; s >= 0; --s)
      for (int w = 0; w < W; ++w) out[kBackProject].push_back({li, rt, s, w});
  for (int rb = 0; rb < (int)ceil_div(L.n, L.ru); ++rb)
    for (int s = 0; s < L.S; ++s) out[kDecompress].push_back({li, rb, s, 0});
}

// HBM bytes a tile of a phase moves (for the queue's lags; approximate).
inline int64_t tile_bytes(const LayerDev& L, int phase, const Tile& t, int W) {
  const int64_t cols = std::min<int64_t>((int64_t)kSeg * 4, (int64_t)L.ld - (int64_t)t.b * kSeg * 4);
  switch (phase) {
    case kProject: return 12 * (int64_t)W * std::min(L.r1, L.n - t.a * L.r1) * cols;
    case kBackProject: return 4 * (int64_t)std::min(L.r3, L.n - t.a * L.r3) * cols;
    case kDecompress: return 4 * (int64_t)std::min(L.ru, L.n - t.a * L.ru) * cols;
    default: return 0;
  }
}

// The fused step's queue: every tile of every phase, in an order where each
// tile's producers come first (project before orthonormalise before
// back-project before decompress, per layer), so that CTAs taking positions
// in order can always finish.  Layers go largest first, so that the last
// dependency chains to drain belong to small layers.  A layer's later phases
// are placed `lag` bytes of other traffic after its previous phase -- about
// what the resident CTAs have in flight -- so that their inputs are usually
// ready when a CTA takes them, while the error state the back-project reads
// is still in L2.  Vector tiles (worker means) go first; with_update false
// leaves out the decompress and vector tiles.
struct QueueStage {
  int layer, phase;
  int64_t ready;  // queue bytes after which the stage's tiles may go in
};

inline std::vector<Tile> build_queue(const std::vector<LayerDev>& hl, const std::vector<Tile>& vec_tiles, int W,
                                     int64_t lag, bool with_update) {
  std::vector<Tile> q;
  auto put = [&](int phase, const Tile& t) {
    Tile x = t;
    x.layer = item_layer(phase, t.layer);
    q.push_back(x);
  };
  if (with_update)
    for (const Tile& t : vec_tiles) put(kItemDecomp, t);
  std::vector<int> order(hl.size());
  for (size_t i = 0; i < hl.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
    return (int64_t)hl[x].n * hl[x].m > (int64_t)hl[y].n * hl[y].m;
  });
  const int last_phase = with_update ? kDecompress : kBackProject;
  std::vector<Tile> tiles[kPhases];
  std::vector<QueueStage> pending;
  int64_t cum = 0;
  std::vector<Tile> stage_tiles[kPhases];
  auto emit_stage = [&](const QueueStage& st) {
    auto& tiles = stage_tiles;
    layer_tiles(hl[st.layer], st.layer, W, tiles);
    int phase = st.phase;
    // orthonormalise and back-project go in together: the orthonormalise
    // tiles are few and short
    const int first = phase, last = (phase == kOrthonormalise) ? kBackProject : phase;
    for (int ph = first; ph <= last; ++ph)
      for (const Tile& t : tiles[ph]) {
        put(ph, t);
        cum += tile_bytes(hl[st.layer], ph, t, W);
      }
    if (last < last_phase) pending.push_back({st.layer, last + 1, cum + lag});
  };
  auto drain = [&](bool all) {
    for (;;) {
      int pick = -1;
      for (size_t i = 0; i < pending.size(); ++i)
        if ((all || pending[i].ready <= cum) && (pick < 0 || pending[i].ready < pending[pick].ready)) pick = (int)i;
      if (pick < 0) return;
      const QueueStage st = pending[pick];
      pending.erase(pending.begin() + pick);
      emit_stage(st);
    }
  };
  for (int li : order) {
    layer_tiles(hl[li], li, W, tiles);
    for (const Tile& t : tiles[kProject]) {
      put(kProject, t);
      cum += tile_bytes(hl[li], kProject, t, W);
      drain(false);
    }
    pending.push_back({li, kOrthonormalise, cum + lag});
    drain(false);
  }
  drain(true);
  return q;
}

}  // namespace psgd
