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
struct TileRows {
  int r1 = 32, r3min = 256, ru = 64;
};

// The phase grids must hold several waves of resident CTAs, or the last,
// partly filled wave leaves HBM idle.
constexpr int kWaves = 4;

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
  const int64_t r3 = std::max<int64_t>(std::max(tr.r3min, 8 * rp), ceil_div(n, 16));
  L.r3 = (int32_t)std::min<int64_t>(n, r3);
  L.t3r = (int32_t)ceil_div(n, L.r3);
  L.c_gram = 0;
  L.c_grp = 1;
  L.c_qs = 1 + L.g1;
  L.c_p3 = L.c_qs + L.S;
  L.c_rb = L.c_p3 + L.S * W;
  return (int64_t)L.c_rb + (L.S > 1 ? L.nrb : 0);
}

// Chooses the tile rows of a layer set so that each phase grid is at least
// kWaves waves of resident CTAs (or the rows reach their floor); decompress
// tiles keep their size (their cost is the per-tile set-up, not the tail).
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
  while (t3 < (int64_t)kWaves * c3 * sms && r.r3min > 32) {
    r.r3min /= 2;
    count(r.r1, r.r3min, r.ru, &t1, &t3, &tu);
  }
  *tr = r;
  return PSGD_OK;
}

}  // namespace psgd
