// psgd_step_noalloc: one PowerSGD step of ONE matrix layer that allocates
// nothing.  The state lives in caller buffers; the scratch (partial P rows,
// Gram partials, R, partial Q_w, counters, the tile lists) lives in one
// file-scope device array of this translation unit whose address is looked
// up once per device.  The phase kernels are the same ones psgd_step runs,
// planned the same way for a one-layer set.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/psgd.h"
#include "psgd_kernels.cuh"
#include "psgd_plan.h"

namespace psgd {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // PSGD_NOALLOC_SCRATCH_BYTES
static_assert(kNoAllocScratchBytes == PSGD_NOALLOC_SCRATCH_BYTES, "header and library disagree");
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

std::atomic<unsigned char*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// First call on a device: the scratch address and the kernels' shared-memory
// limits (both per device).
int scratch_for_device(int dev, unsigned char** out) {
  unsigned char* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      void* addr = nullptr;
      CUDA_TRY(cudaGetSymbolAddress(&addr, g_scratch));
      for (int rp = 1; rp <= 32; rp *= 2) CUDA_TRY(kernels_for(rp)->prepare());
      p = static_cast<unsigned char*>(addr);
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return PSGD_OK;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// Where each piece of the scratch sits (byte offsets) for one layer.
struct ScratchPlan {
  size_t layer, tiles[kPhases], counters, P, gram, rinv, ppart, qpart, total;
  int ntiles[kPhases];
  int ncnt;
};

// Writes the layer record and the tile lists (same order as a context's
// tiles for a one-layer set) and clears the counters, which must start at
// zero.  Grid-stride over every entry.
// W3: back-project tiles per (row tile, segment): W, or 1 when one tile takes
// every worker (the tensor-core back-project).
__global__ void noalloc_tables_kernel(LayerDev L, int W3, LayerDev* dL, Tile* t1, int n1, Tile* tph, int nph,
                                      Tile* t3, int n3, Tile* tu, int nu, unsigned* cnt, int ncnt) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 == 0) *dL = L;
  for (int64_t i = i0; i < ncnt; i += stride) cnt[i] = 0u;
  for (int64_t i = i0; i < n1; i += stride) t1[i] = Tile{0, (int32_t)(i / L.s1), (int32_t)(i % L.s1), 0};
  for (int64_t i = i0; i < nph; i += stride) tph[i] = Tile{0, (int32_t)i, 0, 0};
  for (int64_t i = i0; i < nu; i += stride) tu[i] = Tile{0, (int32_t)(i / L.S), (int32_t)(i % L.S), 0};
  // back-project: last row tile and segment first (the rows project wrote last)
  const int64_t sw = (int64_t)L.S * W3;
  for (int64_t i = i0; i < n3; i += stride)
    t3[i] = Tile{0, (int32_t)(L.t3r - 1 - i / sw), (int32_t)(L.S - 1 - (i / W3) % L.S), (int32_t)(i % W3)};
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace psgd

using namespace psgd;

extern "C" int psgd_step_noalloc(int64_t n, int64_t m, int rank, int num_workers, const float* const* grad_ptrs,
                                 float* B, float* Phat, float* Qbar, float* Qw, float* out_update, int has_prev,
                                 void* cuda_stream) {
  // ---- arguments (host only; nothing is enqueued on a rejection)
  if (n < 1 || n > ((int64_t)1 << 30) || m < 1 || m > ((int64_t)1 << 30))
    return fail(PSGD_ERR_INVALID, "n and m must be in [1, 2^30] (got %lld x %lld)", (long long)n, (long long)m);
  if (rank < 1 || rank > 32 || (rank & (rank - 1)) != 0)
    return fail(PSGD_ERR_INVALID, "rank must be 1, 2, 4, 8, 16 or 32 (got %d)", rank);
  if (rank > n || rank > m)
    return fail(PSGD_ERR_INVALID, "rank %d exceeds min(n, m) = %lld", rank, (long long)std::min(n, m));
  if (num_workers < 1 || num_workers > kMaxWorkers)
    return fail(PSGD_ERR_INVALID, "num_workers must be in [1, %d] (got %d)", kMaxWorkers, num_workers);
  if (!grad_ptrs) return fail(PSGD_ERR_INVALID, "grad_ptrs must not be NULL");
  StepArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int w = 0; w < num_workers; ++w) {
    if (!grad_ptrs[w] || !aligned16(grad_ptrs[w]))
      return fail(PSGD_ERR_INVALID, "grad_ptrs[%d] is NULL or not 16-byte aligned", w);
    a.G[w] = grad_ptrs[w];
  }
  const float* state[4] = {B, Phat, Qbar, Qw};
  const char* names[4] = {"B", "Phat", "Qbar", "Qw"};
  for (int i = 0; i < 4; ++i)
    if (!state[i] || !aligned16(state[i])) return fail(PSGD_ERR_INVALID, "%s is NULL or not 16-byte aligned", names[i]);
  if (out_update && !aligned16(out_update)) return fail(PSGD_ERR_INVALID, "out_update is not 16-byte aligned");

  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(PSGD_ERR_INVALID, "device %d beyond the %d supported", dev, kMaxDevices);
  unsigned char* base = nullptr;
  int rc = scratch_for_device(dev, &base);
  if (rc) return rc;

  // ---- plan: the tiling psgd_create would choose for this one layer
  const int rp = rank;
  const KernelSet* ks = kernels_for(rp);
  const int64_t ld = (m + 3) & ~(int64_t)3;
  const int W = num_workers;
  const std::vector<int64_t> nv{n}, mv{m};
  TileRows tr;
  if ((rc = choose_tile_rows(nv, mv, rp, W, *ks, dev, &tr))) return rc;
  if (ks->mma_rows > 0) {  // the tensor-core project tiles
    tr.r1 = ks->mma_rows;
    tr.pcols = ks->mma_cols;
  }
  const bool bmma = bmma_applies(*ks, W);  // the tensor-core back-project, as a context would
  if (bmma) tr.r3mult = ks->bmma_rows;
  LayerDev L;
  std::memset(&L, 0, sizeof(L));
  ScratchPlan sp;
  sp.ncnt = (int)plan_matrix(L, n, m, ld, rp, W, tr);
  L.off = 0;
  L.index = 0;
  L.p_off = 0;
  L.q_off = 0;
  L.gram_off = 0;
  L.rinv_off = 0;
  L.qpart_off = 0;
  L.ppart_off = 0;
  L.cnt_off = 0;
  sp.ntiles[kProject] = (int)((int64_t)L.nrb * L.s1);
  sp.ntiles[kOrthonormalise] = L.nph;
  sp.ntiles[kBackProject] = (int)((int64_t)L.t3r * L.S * (bmma ? 1 : W));
  sp.ntiles[kDecompress] = (int)(ceil_div(n, L.ru) * L.S);
  const int NG = rp * (rp + 1) / 2;
  size_t pos = 0;
  auto take = [&](size_t bytes) {
    const size_t at = pos;
    pos += round256(bytes);
    return at;
  };
  sp.layer = take(sizeof(LayerDev));
  for (int ph = 0; ph < kPhases; ++ph) sp.tiles[ph] = take((size_t)sp.ntiles[ph] * sizeof(Tile));
  sp.counters = take((size_t)sp.ncnt * sizeof(unsigned));
  sp.P = take((size_t)n * rp * sizeof(float));
  sp.gram = take((size_t)gram_slots(L.nrb, L.g1, L.nph) * NG * sizeof(double));
  sp.rinv = take((size_t)rinv_len(rp) * sizeof(double));
  sp.ppart = take(L.s1 > 1 ? (size_t)L.nrb * L.s1 * L.r1 * rp * sizeof(float) : 0);
  sp.qpart = take((size_t)L.t3r * W * ld * rp * sizeof(float));
  sp.total = pos;
  if (sp.total > kNoAllocScratchBytes)
    return fail(PSGD_ERR_INVALID,
                "layer %lld x %lld at rank %d with %d workers needs %zu bytes of scratch; "
                "psgd_step_noalloc has %zu (use a context: psgd_create)",
                (long long)n, (long long)m, rank, W, sp.total, kNoAllocScratchBytes);

  // ---- enqueue: tables + counters, then the phase kernels
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  LayerDev* dL = reinterpret_cast<LayerDev*>(base + sp.layer);
  Tile* dt[kPhases];
  for (int ph = 0; ph < kPhases; ++ph) dt[ph] = reinterpret_cast<Tile*>(base + sp.tiles[ph]);
  unsigned* cnt = reinterpret_cast<unsigned*>(base + sp.counters);
  noalloc_tables_kernel<<<64, 256, 0, s>>>(L, bmma ? 1 : W, dL, dt[kProject], sp.ntiles[kProject], dt[kOrthonormalise],
                                           sp.ntiles[kOrthonormalise], dt[kBackProject], sp.ntiles[kBackProject],
                                           dt[kDecompress], sp.ntiles[kDecompress], cnt, sp.ncnt);
  CUDA_TRY(cudaGetLastError());
  a.U = out_update;
  a.B = B;
  a.total = n * ld;
  a.P = reinterpret_cast<float*>(base + sp.P);
  a.Phat = Phat;
  a.Qbar = Qbar;
  a.Qw = Qw;
  a.q_total = ld * rp;
  a.gram = reinterpret_cast<double*>(base + sp.gram);
  a.rinv = reinterpret_cast<double*>(base + sp.rinv);
  a.qpart = reinterpret_cast<float*>(base + sp.qpart);
  a.ppart = reinterpret_cast<float*>(base + sp.ppart);
  a.counters = cnt;
  a.layers = dL;
  a.vecs = nullptr;
  a.W = W;
  a.qbar_scale = 1.0f / (float)W;
  a.has_prev = has_prev ? 1 : 0;
  a.stall_layer = -1;
  const int phases = out_update ? kPhases : kPhases - 1;
  for (int ph = 0; ph < phases; ++ph) {
    if (sp.ntiles[ph] == 0) continue;
    a.tiles = dt[ph];
    if (ph == kBackProject && bmma)
      CUDA_TRY(ks->launch_bmma(a, sp.ntiles[ph], s));
    else
      CUDA_TRY(ks->launch(ph, a, sp.ntiles[ph], s));
  }
  return PSGD_OK;
}
