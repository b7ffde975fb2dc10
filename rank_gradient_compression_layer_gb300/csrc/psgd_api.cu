// Host side of libpsgd.so: the C ABI declared in include/psgd.h.
//
// psgd_create plans the packed layout and the tiles of the four phase kernels
// (project, orthonormalise, back-project, decompress), owns every device
// buffer of the state and initialises Q.  psgd_step fills a StepArgs and
// enqueues the four kernels on the context's stream; nothing else runs on the
// host per step.
#define PSGD_SIDE_KERNELS 1

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/psgd.h"
#include "psgd_dispatch.h"
#include "psgd_kernels.cuh"
#include "psgd_plan.h"
#include "psgd_rtopk.h"

using namespace psgd;

namespace {
thread_local std::string g_err;

// NVTX ranges on the host timeline, one per step and one per phase launch
// (no-ops unless a profiling tool is attached).
const char* const kPhaseRange[kPhases] = {"psgd project", "psgd orthonormalise", "psgd back-project",
                                          "psgd decompress"};
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace

namespace psgd {

int fail(int code, const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  const int code = (e == cudaErrorMemoryAllocation) ? PSGD_ERR_OOM : PSGD_ERR_CUDA;
  return fail(code, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace psgd

namespace {

int check_layers(int num_layers, const int64_t* n, const int64_t* m) {
  if (num_layers < 1) return fail(PSGD_ERR_INVALID, "num_layers must be >= 1 (got %d)", num_layers);
  if (!n || !m) return fail(PSGD_ERR_INVALID, "n and m must not be NULL");
  for (int l = 0; l < num_layers; ++l) {
    if (n[l] < 1 || n[l] > (int64_t)1 << 30)
      return fail(PSGD_ERR_INVALID, "layer %d: n = %lld out of range [1, 2^30]", l, (long long)n[l]);
    if (m[l] < 0 || m[l] > (int64_t)1 << 30)
      return fail(PSGD_ERR_INVALID, "layer %d: m = %lld out of range [0, 2^30]", l, (long long)m[l]);
    if (m[l] > 0 && n[l] * m[l] > ((int64_t)1 << 40))
      return fail(PSGD_ERR_INVALID, "layer %d: n*m too large", l);
  }
  return PSGD_OK;
}

// Packed layout: 16-byte aligned layers, matrix rows padded to a multiple of 4.
void layout(int num_layers, const int64_t* n, const int64_t* m, int64_t* off, int64_t* ld, int64_t* total) {
  int64_t pos = 0;
  for (int l = 0; l < num_layers; ++l) {
    off[l] = pos;
    if (m[l] > 0) {
      ld[l] = (m[l] + 3) & ~(int64_t)3;
      pos += n[l] * ld[l];
    } else {
      ld[l] = 0;
      pos += (n[l] + 3) & ~(int64_t)3;
    }
  }
  *total = pos;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Seed of step t's fresh Q in the unbiased variant: the splitmix64 output
// function (Steele, Lea & Flood 2014) of seed + (t + 1) * golden gamma.
uint64_t step_seed(uint64_t seed, int64_t step) {
  uint64_t z = seed + (uint64_t)(step + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Packs Phat (n x r out of n x RP) and Qbar (m x r out of ld x RP) of every
// matrix layer into one contiguous message: the floats a worker would send.
struct PackEntry {
  int64_t src_p, src_q, dst;
  int32_t n, m;
};

__global__ void pack_msg_kernel(float* dst, const float* Phat, const float* Qbar, const PackEntry* ent, int r,
                                int rp) {
  const PackEntry e = ent[blockIdx.y];
  const int64_t np = (int64_t)e.n * r, nq = (int64_t)e.m * r;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < np + nq;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v;
    if (i < np)
      v = Phat[e.src_p + (i / r) * rp + (i % r)];
    else
      v = Qbar[e.src_q + ((i - np) / r) * rp + ((i - np) % r)];
    dst[e.dst + i] = v;
  }
}

// One layer's block in an exchange buffer of the split step: the dense
// rows x r block at dense_off <-> rows x RP at pad_off of P or Qbar (vec = 0),
// or a vector layer's n floats <-> the packed gradient offset pad_off (vec = 1).
struct XEntry {
  int64_t pad_off, dense_off;
  int32_t rows, vec;
};

// Split step exchange.  to_dense: matrix blocks from `padded` into `dense`;
// vector blocks get qbar_scale * the sum of this process's gradients (their
// share of the all-reduced mean).  !to_dense: matrix blocks from `dense` into
// `padded`; vector blocks into the update a.U (when not NULL).  One
// blockIdx.y per entry.
__global__ void xchg_kernel(const StepArgs a, float* dense, float* padded, const XEntry* ent, int r, int rp,
                            int to_dense) {
  const XEntry e = ent[blockIdx.y];
  const int64_t cnt = e.vec ? (int64_t)e.rows : (int64_t)e.rows * r;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < cnt; i += (int64_t)gridDim.x * blockDim.x) {
    if (e.vec) {
      if (to_dense) {
        float sum = 0.f;
        for (int w = 0; w < a.W; ++w) sum += a.G[w][e.pad_off + i];
        dense[e.dense_off + i] = sum * a.qbar_scale;
      } else if (a.U) {
        a.U[e.pad_off + i] = dense[e.dense_off + i];
      }
      continue;
    }
    float* pp = padded + e.pad_off + (i / r) * rp + (i % r);
    if (to_dense)
      dense[e.dense_off + i] = *pp;
    else
      *pp = dense[e.dense_off + i];
  }
}

}  // namespace

struct psgd_ctx {
  int device = 0;
  cudaStream_t stream = nullptr;
  int num_layers = 0, rank = 0, rp = 0, W = 0;
  uint64_t seed = 0;
  const KernelSet* ks = nullptr;
  std::vector<int64_t> n, m, off, ld;
  std::vector<int> mat_of;  // layer -> matrix index or -1
  std::vector<LayerDev> hl;
  std::vector<VecDev> hv;
  std::vector<Tile> tiles[kPhases];
  std::vector<PackEntry> pack;
  int64_t total = 0, q_total = 0, p_total = 0, gram_total = 0, rinv_total = 0, qpart_total = 0,
          ppart_total = 0;
  int64_t n_counters = 0, msg_floats = 0;
  // device state and scratch
  float *B = nullptr, *P = nullptr, *Phat = nullptr, *Qbar = nullptr, *Qw = nullptr, *qpart = nullptr,
        *ppart = nullptr;
  double *gram = nullptr, *rinv = nullptr;
  unsigned* counters = nullptr;
  LayerDev* d_layers = nullptr;
  VecDev* d_vecs = nullptr;
  Tile* d_tiles[kPhases] = {nullptr, nullptr, nullptr, nullptr};
  PackEntry* d_pack = nullptr;
  // lazily allocated: error read-back scratch, host-path staging
  float* e_scratch = nullptr;
  int64_t e_scratch_elems = 0;
  float *stage_G = nullptr, *stage_U = nullptr, *stage_msg = nullptr;
  // optional phase timing: one set of kPhases + 1 events per step, in a ring
  bool timing = false;
  std::vector<cudaEvent_t> ev;  // kTimedSteps x (kPhases + 1)
  int64_t timed_since = 0;      // steps recorded since the last psgd_get_phase_times
  int tile_rows[3] = {0, 0, 0};  // project rows, least back-project rows, decompress rows
  int has_prev = 0;
  bool unbiased = false;  // psgd_options.unbiased: fresh shared Q per step, no error feedback
  RTopK* rk = nullptr;    // psgd_options.compressor == PSGD_RTOPK: the rTop-k plan
  int top_div = 0, sample_div = 0;
  bool broken = false;
  // the fused step (padded rank <= 4, PowerSGD): queues without [0] and with
  // [1] the decompress tiles, flags, ticket / status words, CTAs per launch
  bool fused = false;
  std::vector<Tile> queue[2];
  Tile* d_queue[2] = {nullptr, nullptr};
  unsigned* flags = nullptr;
  unsigned* sync_words = nullptr;
  int64_t n_flags = 0;
  int fused_ctas = 0;
  int64_t wait_ns = 2000000000LL;
  int stall_layer = -1;
  // the split step (psgd_step_begin / mid / end): workers over all
  // processes, where the step stands (0 idle, 1 after begin, 2 after mid),
  // the gradients of begin, the Gram tiles, the decompress tiles of the
  // matrix layers, and the exchange layouts of P and of Q (+ vector sums)
  int total_workers = 0;
  int split_phase = 0;
  std::vector<const float*> split_grads;
  std::vector<Tile> gram_tiles, mat_u_tiles;
  std::vector<XEntry> xp, xq;
  Tile *d_gram_tiles = nullptr, *d_mat_u_tiles = nullptr;
  XEntry *d_xp = nullptr, *d_xq = nullptr;
  int64_t xp_floats = 0, xq_floats = 0;
  // the one-pass project (psgd_step at padded rank <= 4): cluster items over
  // the layers' row groups, and the Y partials they write
  bool bmma = false;  // the back-project runs on the tensor cores (tiles without a worker)
  bool ypath = false;
  std::vector<Tile> ytiles;  // y_clusters header tiles, then the segments
  Tile* d_ytiles = nullptr;
  int y_clusters = 0;
  size_t y_smem = 0;
  float* ypart = nullptr;
  int64_t y_total = 0;
  // stats
  int64_t steps = 0, sent_step = 0, unc_step = 0, mat_el = 0, vec_el = 0;
};

namespace {

void free_all(psgd_ctx* c) {
  void* ptrs[] = {c->B, c->P, c->Phat, c->Qbar, c->Qw, c->qpart, c->ppart, c->gram, c->rinv, c->counters,
                  c->d_layers, c->d_vecs, c->d_tiles[0], c->d_tiles[1], c->d_tiles[2], c->d_tiles[3], c->d_pack,
                  c->e_scratch, c->stage_G, c->stage_U, c->stage_msg, c->d_queue[0], c->d_queue[1], c->flags,
                  c->sync_words, c->d_gram_tiles, c->d_mat_u_tiles, c->d_xp, c->d_xq, c->d_ytiles, c->ypart};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  rtopk_destroy(c->rk);
  c->rk = nullptr;
  for (cudaEvent_t e : c->ev)
    if (e) cudaEventDestroy(e);
  c->ev.clear();
}

template <class T>
int dalloc(T** p, int64_t count, const char* what) {
  if (count <= 0) count = 1;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), (size_t)count * sizeof(T));
  if (e != cudaSuccess) {
    *p = nullptr;
    return cuda_fail(e, what);
  }
  return PSGD_OK;
}

// The one-pass project's plan: per layer the column split; the dynamic
// shared memory of the Y accumulators (the largest layer's need); the
// clusters that fit on the GPU at once with it, each given an equal share of
// the layers' row blocks (plan_yschedule); per layer the counters, Gram and Y
// partial slots.  Leaves c->ypath false when a layer does not fit or no
// cluster fits on the GPU.
void plan_one_pass(psgd_ctx* c) {
  int64_t smem = 0;
  for (LayerDev& L : c->hl) {
    if (!plan_ycols(L, c->rp, c->W)) c->ypath = false;
    else smem = std::max(smem, y_smem_bytes((int64_t)L.yfc * c->W, c->rp));
  }
  int clusters = 0;
  if (c->ypath &&
      (c->ks->occupancy_cluster(kYClusterMax, (size_t)smem, &clusters) != cudaSuccess || clusters <= 0)) {
    cudaGetLastError();
    c->ypath = false;
  }
  if (!c->ypath) {
    for (LayerDev& L : c->hl) L.cw = L.yfc = 0;
    return;
  }
  c->y_smem = (size_t)smem;
  c->y_clusters = clusters;
  plan_yschedule(c->hl, c->rp, c->W, clusters, c->ytiles);
  const int rp = c->rp, NG = rp * (rp + 1) / 2;
  for (LayerDev& L : c->hl) {
    L.c_yg = (int32_t)(c->n_counters - L.cnt_off);
    c->n_counters += ceil_div(L.nys, kGramGroup);
    L.ygram_off = c->gram_total;
    c->gram_total += (L.nys + ceil_div(L.nys, kGramGroup)) * NG;
    L.y_off = c->y_total;
    c->y_total += (int64_t)L.nys * c->W * L.ld * rp;
  }
}

// The order of the matrix layers in the project and back-project phases:
// largest first (stable), so that each grid ends on the short tiles of small
// layers, and the long closing sums of the large layers (their row blocks'
// segment and Gram partials, their segments' Q_w sums) overlap other
// layers' streaming instead of trailing the phase.
std::vector<int> layer_order(const psgd_ctx* c) {
  std::vector<int> order(c->hl.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
    return (int64_t)c->hl[x].n * c->hl[x].ld > (int64_t)c->hl[y].n * c->hl[y].ld;
  });
  return order;
}

// The error rows the back-project reads first (the first layers' last rows:
// it takes each layer's row tiles from the last): up to kL2KeepShare of L2,
// counted from the start of the layer order, are stored by the project phase
// with an L2 evict-last policy so that they are still there.
void plan_l2_keep(psgd_ctx* c) {
  int l2 = 0;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, c->device) != cudaSuccess) {
    cudaGetLastError();
    l2 = 0;
  }
  int64_t room = (int64_t)(kL2KeepShare * (double)l2);
  for (int li : layer_order(c)) {
    LayerDev& L = c->hl[li];
    const int64_t row_bytes = (int64_t)c->W * L.ld * 4;
    const int64_t rows = std::min<int64_t>(L.n, std::max<int64_t>(0, room / row_bytes));
    L.l2row = (int32_t)(L.n - rows);
    room -= rows * row_bytes;
  }
}

// Tiles of every phase.  Project and back-project take the layers in
// layer_order; the back-project takes a layer's row tiles from the last, so
// it starts on rows the project phase kept in L2.
void build_tiles(psgd_ctx* c) {
  for (auto& v : c->tiles) v.clear();
  const int nm = (int)c->hl.size();
  const std::vector<int> order = layer_order(c);
  for (int li : order) {
    const LayerDev& L = c->hl[li];
    for (int rb = 0; rb < L.nrb; ++rb)
      for (int s = 0; s < L.s1; ++s) c->tiles[kProject].push_back({li, rb, s, 0});
  }
  for (int li = 0; li < nm; ++li) {
    const LayerDev& L = c->hl[li];
    for (int t = 0; t < L.nph; ++t) c->tiles[kOrthonormalise].push_back({li, t, 0, 0});
    for (int rb = 0; rb < (int)ceil_div(L.n, L.ru); ++rb)
      for (int s = 0; s < L.S; ++s) c->tiles[kDecompress].push_back({li, rb, s, 0});
  }
  for (int li : order) {
    const LayerDev& L = c->hl[li];
    for (int rt = L.t3r - 1; rt >= 0; --rt)
      for (int s = L.S - 1; s >= 0; --s)
        for (int w = 0; w < (c->bmma ? 1 : c->W); ++w) c->tiles[kBackProject].push_back({li, rt, s, w});
  }
  for (int vi = 0; vi < (int)c->hv.size(); ++vi)
    for (int t = 0; t < (int)ceil_div(c->hv[vi].n, kVChunk); ++t) c->tiles[kDecompress].push_back({vi, t, 0, 1});
}

constexpr int kTimedSteps = 256;  // steps whose phase times one psgd_get_phase_times can average

int ctx_ok(const psgd_ctx* c) {
  if (!c) return fail(PSGD_ERR_INVALID, "context is NULL");
  if (c->broken) return fail(PSGD_ERR_STATE, "context hit an earlier CUDA error; destroy it");
  return PSGD_OK;
}

int matrix_layer(const psgd_ctx* c, int layer, const LayerDev** L) {
  if (layer < 0 || layer >= c->num_layers) return fail(PSGD_ERR_INVALID, "layer %d out of range", layer);
  const int mi = c->mat_of[layer];
  if (mi < 0) return fail(PSGD_ERR_INVALID, "layer %d is a vector layer", layer);
  *L = &c->hl[mi];
  return PSGD_OK;
}

int sync_and_check(psgd_ctx* c) {
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) {
    c->broken = true;
    return cuda_fail(e, "step");
  }
  if (c->steps > 0) {
    unsigned status = 0;
    e = cudaMemcpy(&status, c->sync_words + 2, sizeof(status), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      c->broken = true;
      return cuda_fail(e, "step status");
    }
    if (status == 2) {
      c->broken = true;
      return fail(PSGD_ERR_TIMEOUT, "a step was abandoned: a wait for the tensor cores ran out");
    }
    if (status != 0) {
      c->broken = true;
      return fail(PSGD_ERR_TIMEOUT, "a fused step was abandoned: a tile waited longer than %lld ms for its inputs",
                  (long long)(c->wait_ns / 1000000));
    }
  }
  return PSGD_OK;
}

// Tiles per layer phase and the fused queues of a context (all matrix
// layers and vector chunks, with and without the decompress tiles).
void build_queues(psgd_ctx* c, int64_t lag) {
  std::vector<Tile> vec_tiles;
  for (const Tile& t : c->tiles[kDecompress])
    if (t.c == 1) vec_tiles.push_back(t);
  c->queue[0] = build_queue(c->hl, vec_tiles, c->W, lag, false);
  c->queue[1] = build_queue(c->hl, vec_tiles, c->W, lag, true);
}

// The default lag between a layer's phases in the fused queue: twice what
// the resident CTAs of the fused step have in flight, one average project
// tile each.
int64_t default_lag(const psgd_ctx* c, int ctas) {
  int64_t bytes = 0;
  for (const Tile& t : c->tiles[kProject]) bytes += tile_bytes(c->hl[t.layer], kProject, t, c->W);
  const int64_t nt = std::max<int64_t>(1, (int64_t)c->tiles[kProject].size());
  return 2 * (int64_t)ctas * (bytes / nt);
}

}  // namespace

extern "C" {

const char* psgd_last_error(void) { return g_err.c_str(); }

const char* psgd_version(void) { return "psgd 0.2 (sm_103a)"; }

int psgd_plan_layout(int num_layers, const int64_t* n, const int64_t* m, int64_t* offset, int64_t* ld,
                     int64_t* total) {
  int rc = check_layers(num_layers, n, m);
  if (rc) return rc;
  if (!offset || !ld || !total) return fail(PSGD_ERR_INVALID, "output pointers must not be NULL");
  layout(num_layers, n, m, offset, ld, total);
  return PSGD_OK;
}

int psgd_count_sent(int num_layers, const int64_t* n, const int64_t* m, int rank, int64_t* compressed,
                    int64_t* uncompressed) {
  int rc = check_layers(num_layers, n, m);
  if (rc) return rc;
  if (rank < 1) return fail(PSGD_ERR_INVALID, "rank must be >= 1");
  if (!compressed || !uncompressed) return fail(PSGD_ERR_INVALID, "output pointers must not be NULL");
  int64_t cs = 0, us = 0;
  for (int l = 0; l < num_layers; ++l) {
    if (m[l] == 0) {
      cs += n[l];
      us += n[l];
    } else {
      cs += (n[l] + m[l]) * rank;
      us += n[l] * m[l];
    }
  }
  *compressed = cs;
  *uncompressed = us;
  return PSGD_OK;
}

int psgd_plan_one_pass(int num_layers, const int64_t* n, const int64_t* m, int rank, int num_workers,
                       int clusters, int32_t* layer_plan, int32_t* tiles, int64_t* count) {
  int rc = check_layers(num_layers, n, m);
  if (rc) return rc;
  if (rank < 1 || rank > 4) return fail(PSGD_ERR_INVALID, "the one-pass project is for ranks 1..4 (got %d)", rank);
  if (num_workers < 1 || num_workers > kMaxWorkers)
    return fail(PSGD_ERR_INVALID, "num_workers must be in [1, %d] (got %d)", kMaxWorkers, num_workers);
  if (clusters < 1) return fail(PSGD_ERR_INVALID, "clusters must be >= 1 (got %d)", clusters);
  if (!count) return fail(PSGD_ERR_INVALID, "count must not be NULL");
  const int rp = padded_rank(rank);
  std::vector<int64_t> off(num_layers), ld(num_layers);
  int64_t total = 0;
  layout(num_layers, n, m, off.data(), ld.data(), &total);
  std::vector<LayerDev> hl;
  for (int l = 0; l < num_layers; ++l) {
    if (m[l] == 0) continue;
    LayerDev L;
    std::memset(&L, 0, sizeof(L));
    L.n = (int32_t)n[l];
    L.F = (int32_t)(ld[l] / 4);
    L.ld = (int32_t)ld[l];
    if (!plan_ycols(L, rp, num_workers)) return fail(PSGD_ERR_INVALID, "layer %d does not fit the one-pass project", l);
    hl.push_back(L);
  }
  std::vector<Tile> t;
  plan_yschedule(hl, rp, num_workers, clusters, t);
  *count = (int64_t)t.size();
  if (layer_plan)
    for (size_t i = 0; i < hl.size(); ++i) {
      layer_plan[4 * i] = hl[i].cw;
      layer_plan[4 * i + 1] = hl[i].yfc;
      layer_plan[4 * i + 2] = hl[i].yr;
      layer_plan[4 * i + 3] = hl[i].nys;
    }
  if (tiles)
    for (size_t i = 0; i < t.size(); ++i) {
      tiles[4 * i] = t[i].layer;
      tiles[4 * i + 1] = t[i].a;
      tiles[4 * i + 2] = t[i].b;
      tiles[4 * i + 3] = t[i].c;
    }
  return PSGD_OK;
}

int psgd_plan_queue(int num_layers, const int64_t* n, const int64_t* m, int rank, int num_workers,
                    int project_rows, int64_t lag_bytes, int with_update, int32_t* items, int64_t* count) {
  int rc = check_layers(num_layers, n, m);
  if (rc) return rc;
  if (rank < 1 || rank > 32) return fail(PSGD_ERR_INVALID, "rank must be in [1, 32] (got %d)", rank);
  if (num_workers < 1 || num_workers > kMaxWorkers)
    return fail(PSGD_ERR_INVALID, "num_workers must be in [1, %d] (got %d)", kMaxWorkers, num_workers);
  if (!count) return fail(PSGD_ERR_INVALID, "count must not be NULL");
  const int rp = padded_rank(rank);
  const KernelSet* ks = kernels_for(rp);
  if (project_rows < 0 || project_rows > ks->r1) return fail(PSGD_ERR_INVALID, "project_rows out of range");
  TileRows tr;
  tr.r1 = project_rows > 0 ? project_rows : ks->r1;
  tr.ru = ks->ru;
  std::vector<int64_t> off(num_layers), ld(num_layers);
  int64_t total = 0;
  layout(num_layers, n, m, off.data(), ld.data(), &total);
  std::vector<LayerDev> hl;
  std::vector<Tile> vec_tiles;
  int nv = 0;
  for (int l = 0; l < num_layers; ++l) {
    if (m[l] == 0) {
      for (int t = 0; t < (int)ceil_div(n[l], kVChunk); ++t) vec_tiles.push_back({nv, t, 0, 1});
      ++nv;
      continue;
    }
    LayerDev L;
    std::memset(&L, 0, sizeof(L));
    plan_matrix(L, n[l], m[l], ld[l], rp, num_workers, tr);
    L.index = l;
    hl.push_back(L);
  }
  const std::vector<Tile> q = build_queue(hl, vec_tiles, num_workers, std::max<int64_t>(0, lag_bytes), with_update != 0);
  *count = (int64_t)q.size();
  if (items)
    for (size_t i = 0; i < q.size(); ++i) {
      items[4 * i] = q[i].layer;
      items[4 * i + 1] = q[i].a;
      items[4 * i + 2] = q[i].b;
      items[4 * i + 3] = q[i].c;
    }
  return PSGD_OK;
}

int psgd_create(psgd_ctx** out, int num_layers, const int64_t* n, const int64_t* m, int rank, int num_workers,
                uint64_t seed, void* cuda_stream) {
  return psgd_create_ex(out, num_layers, n, m, rank, num_workers, seed, cuda_stream, nullptr);
}

int psgd_create_ex(psgd_ctx** out, int num_layers, const int64_t* n, const int64_t* m, int rank,
                   int num_workers, uint64_t seed, void* cuda_stream, const psgd_options* opt) {
  if (!out) return fail(PSGD_ERR_INVALID, "out must not be NULL");
  *out = nullptr;
  int rc = check_layers(num_layers, n, m);
  if (rc) return rc;
  if (rank < 1 || rank > 32) return fail(PSGD_ERR_INVALID, "rank must be in [1, 32] (got %d)", rank);
  if (num_workers < 1 || num_workers > kMaxWorkers)
    return fail(PSGD_ERR_INVALID, "num_workers must be in [1, %d] (got %d)", kMaxWorkers, num_workers);
  for (int l = 0; l < num_layers; ++l)
    if (m[l] > 0 && (rank > n[l] || rank > m[l]))
      return fail(PSGD_ERR_INVALID, "layer %d: rank %d exceeds min(n, m) = %lld", l, rank,
                  (long long)std::min(n[l], m[l]));

  psgd_ctx* c = new psgd_ctx();
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  c->num_layers = num_layers;
  c->rank = rank;
  c->rp = padded_rank(rank);
  c->W = num_workers;
  c->seed = seed;
  c->ks = kernels_for(c->rp);
  c->timing = opt && opt->timing;
  c->unbiased = opt && opt->unbiased;
  c->total_workers = (opt && opt->total_workers > 0) ? opt->total_workers : num_workers;
  const bool rtopk = opt && opt->compressor == PSGD_RTOPK;
  if (opt && opt->compressor != PSGD_POWERSGD && !rtopk) {
    delete c;
    return fail(PSGD_ERR_INVALID, "unknown compressor %d", opt->compressor);
  }
  if (rtopk && (c->unbiased || opt->rtopk_top_div < 1 || opt->rtopk_sample_div < 1)) {
    delete c;
    return fail(PSGD_ERR_INVALID, "rTop-k needs top_div, sample_div >= 1 and no unbiased option");
  }
  if (rtopk) {
    c->top_div = opt->rtopk_top_div;
    c->sample_div = opt->rtopk_sample_div;
  }
  if (c->total_workers < num_workers || (c->total_workers != num_workers && (rtopk || c->unbiased))) {
    delete c;
    return fail(PSGD_ERR_INVALID, "total_workers must be >= num_workers, and is for PowerSGD only");
  }
  if (cudaGetDevice(&c->device) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return fail(PSGD_ERR_CUDA, "no CUDA device");
  }
  c->n.assign(n, n + num_layers);
  c->m.assign(m, m + num_layers);
  c->off.resize(num_layers);
  c->ld.resize(num_layers);
  layout(num_layers, n, m, c->off.data(), c->ld.data(), &c->total);
  c->mat_of.assign(num_layers, -1);

  const int rp = c->rp;
  const int NG = rp * (rp + 1) / 2;
  TileRows tr;
  // the kernels' shared-memory limits first: the occupancy the tile planner
  // reads depends on them (above 48 KB of dynamic shared memory a kernel
  // reports no resident CTAs until its limit is raised)
  {
    cudaError_t e = c->ks->prepare();
    if (e != cudaSuccess) {
      delete c;
      return cuda_fail(e, "kernel attributes");
    }
  }
  if ((rc = choose_tile_rows(c->n, c->m, rp, c->W, *c->ks, c->device, &tr))) {
    delete c;
    return rc;
  }
  // the fused step takes its tiles from a queue, with no phase tail to fill:
  // the largest project tiles halve the number of tiles it runs
  if (c->ks->launch_fused && !c->unbiased && !rtopk && opt && opt->fused && c->total_workers == c->W)
    tr.r1 = c->ks->r1;
  const bool mma = c->ks->mma_rows > 0 && !c->unbiased && !rtopk;
  if (mma && opt && opt->project_rows > 0) {
    delete c;
    return fail(PSGD_ERR_INVALID, "project_rows is fixed at %d rows for the tensor-core project tiles", c->ks->mma_rows);
  }
  if (mma) {
    tr.r1 = c->ks->mma_rows;
    tr.pcols = c->ks->mma_cols;
  }
  // the back-project on the tensor cores (r = 32: at r = 16 the CUDA-core
  // kernel is faster): every worker's D in TMEM (W r <= 512 columns), row
  // tiles in whole chunks
  c->bmma = bmma_applies(*c->ks, c->W) && !c->unbiased && !rtopk;
  if (c->bmma) tr.r3mult = c->ks->bmma_rows;
  if (opt && opt->project_rows > 0) {
    if (opt->project_rows > c->ks->r1 || opt->project_rows % c->ks->rsb != 0) {
      delete c;
      return fail(PSGD_ERR_INVALID, "project_rows must be a multiple of %d and <= %d", c->ks->rsb, c->ks->r1);
    }
    tr.r1 = opt->project_rows;
  }
  c->tile_rows[0] = tr.r1;
  c->tile_rows[1] = tr.r3min;
  c->tile_rows[2] = tr.ru;
  for (int l = 0; l < num_layers; ++l) {
    if (m[l] == 0) {
      c->hv.push_back({c->off[l], (int32_t)n[l], 0});
      c->vec_el += n[l];
      c->sent_step += n[l];
      c->unc_step += n[l];
      continue;
    }
    LayerDev L;
    std::memset(&L, 0, sizeof(L));
    const int64_t ncnt = plan_matrix(L, n[l], m[l], c->ld[l], rp, c->W, tr);
    L.off = c->off[l];
    L.index = l;
    L.p_off = c->p_total;
    c->p_total += (n[l] * rp + 3) & ~(int64_t)3;
    L.q_off = c->q_total;
    c->q_total += c->ld[l] * rp;
    L.gram_off = c->gram_total;
    c->gram_total += gram_slots(L.nrb, L.g1, L.nph) * NG;
    L.rinv_off = c->rinv_total;
    c->rinv_total += rinv_len(rp);
    L.qpart_off = c->qpart_total;
    c->qpart_total += (int64_t)L.t3r * c->W * c->ld[l] * rp;
    L.ppart_off = c->ppart_total;
    if (L.s1 > 1) c->ppart_total += (int64_t)L.nrb * L.s1 * L.r1 * rp;
    L.cnt_off = (int32_t)c->n_counters;
    c->n_counters += ncnt;
    L.f_off = (int32_t)c->n_flags;
    c->n_flags += kFlagQbar + L.S;
    // the message: Phat and Qbar; the unbiased variant sends P alone;
    // rTop-k: k indices and k values per worker
    int64_t sent = c->unbiased ? n[l] * rank : (n[l] + m[l]) * rank;
    if (rtopk) sent = 2 * ceil_div(ceil_div(n[l] * m[l], c->top_div), c->sample_div);
    c->pack.push_back({L.p_off, L.q_off, c->msg_floats, L.n, c->unbiased ? 0 : L.m});
    c->msg_floats += rtopk ? sent * num_workers : sent;
    c->mat_of[l] = (int)c->hl.size();
    c->hl.push_back(L);
    c->mat_el += n[l] * m[l];
    c->sent_step += sent;
    c->unc_step += n[l] * m[l];
  }
  build_tiles(c);
  plan_l2_keep(c);
  // the one-pass project (options.one_pass): PowerSGD at padded rank <= 4,
  // every worker in this process, four phase kernels
  c->ypath = c->ks->launch_cluster && !c->unbiased && !rtopk && opt && opt->one_pass > 0 && !opt->fused &&
             !c->hl.empty() && c->total_workers == c->W;
  if (c->ypath) plan_one_pass(c);
  // the fused step: PowerSGD at padded rank <= 4 with at least one matrix
  c->fused = c->ks->launch_fused && !c->unbiased && !rtopk && opt && opt->fused && !c->hl.empty() &&
             c->total_workers == c->W;
  // the split step's tiles and exchange layouts
  for (const Tile& t : c->tiles[kProject])
    if (t.b == 0) c->gram_tiles.push_back(t);
  for (const Tile& t : c->tiles[kDecompress])
    if (t.c == 0) c->mat_u_tiles.push_back(t);
  for (int l = 0; l < num_layers; ++l) {
    if (m[l] == 0) continue;
    const LayerDev& L = c->hl[c->mat_of[l]];
    c->xp.push_back({L.p_off, c->xp_floats, L.n, 0});
    c->xp_floats += (int64_t)L.n * rank;
    c->xq.push_back({L.q_off, c->xq_floats, L.m, 0});
    c->xq_floats += (int64_t)L.m * rank;
  }
  for (int l = 0; l < num_layers; ++l)
    if (m[l] == 0) {
      c->xq.push_back({c->off[l], c->xq_floats, (int32_t)n[l], 1});
      c->xq_floats += n[l];
    }
  if (opt && opt->wait_ms > 0) c->wait_ns = (int64_t)opt->wait_ms * 1000000;
  if (opt && opt->test_stall > 0 && !c->hl.empty())
    c->stall_layer = c->hl[std::min<int>(opt->test_stall - 1, (int)c->hl.size() - 1)].index;
  if (c->fused) {
    int per_sm = 0, sms = 0;
    cudaError_t e = c->ks->occupancy_fused(&per_sm);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
      delete c;
      return cuda_fail(e, "fused step occupancy");
    }
    const int resident = std::max(1, per_sm * sms);
    const int64_t lag = (opt && opt->queue_lag_kb > 0) ? (int64_t)opt->queue_lag_kb * 1024 : default_lag(c, resident);
    build_queues(c, lag);
    c->fused_ctas = resident;
  }

  const int W = c->W;
  rc = PSGD_OK;
#define ALLOC(p, cnt) \
  if (!rc) rc = dalloc(&c->p, (cnt), #p)
  ALLOC(B, (int64_t)W * c->total);
  ALLOC(P, c->p_total);
  ALLOC(Phat, c->p_total);
  ALLOC(Qbar, c->q_total);
  ALLOC(Qw, (int64_t)W * c->q_total);
  ALLOC(qpart, c->qpart_total);
  ALLOC(ppart, c->ppart_total);
  ALLOC(gram, c->gram_total);
  ALLOC(rinv, c->rinv_total);
  ALLOC(counters, c->n_counters);
  ALLOC(d_layers, (int64_t)c->hl.size());
  ALLOC(d_vecs, (int64_t)c->hv.size());
  for (int ph = 0; ph < kPhases; ++ph) ALLOC(d_tiles[ph], (int64_t)c->tiles[ph].size());
  ALLOC(d_pack, (int64_t)c->pack.size());
  ALLOC(d_gram_tiles, (int64_t)c->gram_tiles.size());
  ALLOC(d_mat_u_tiles, (int64_t)c->mat_u_tiles.size());
  ALLOC(d_xp, (int64_t)c->xp.size());
  ALLOC(d_xq, (int64_t)c->xq.size());
  ALLOC(sync_words, 4);
  ALLOC(ypart, c->y_total);
  ALLOC(d_ytiles, (int64_t)c->ytiles.size());
  if (c->fused) {
    ALLOC(d_queue[0], (int64_t)c->queue[0].size());
    ALLOC(d_queue[1], (int64_t)c->queue[1].size());
    ALLOC(flags, c->n_flags);
  }
#undef ALLOC
  if (rc) {
    free_all(c);
    delete c;
    return rc;
  }
  auto setup = [&]() -> int {
    cudaStream_t s = c->stream;
    if (c->timing) {
      c->ev.assign((size_t)kTimedSteps * (kPhases + 1), nullptr);
      for (auto& e : c->ev) CUDA_TRY(cudaEventCreate(&e));
    }
    CUDA_TRY(cudaMemsetAsync(c->B, 0, (size_t)W * c->total * sizeof(float), s));
    CUDA_TRY(cudaMemsetAsync(c->Phat, 0, (size_t)std::max<int64_t>(c->p_total, 1) * sizeof(float), s));
    CUDA_TRY(cudaMemsetAsync(c->Qbar, 0, (size_t)std::max<int64_t>(c->q_total, 1) * sizeof(float), s));
    CUDA_TRY(cudaMemsetAsync(c->Qw, 0, (size_t)std::max<int64_t>(W * c->q_total, 1) * sizeof(float), s));
    CUDA_TRY(cudaMemsetAsync(c->counters, 0, (size_t)std::max<int64_t>(c->n_counters, 1) * sizeof(unsigned), s));
    CUDA_TRY(cudaMemsetAsync(c->rinv, 0, (size_t)std::max<int64_t>(c->rinv_total, 1) * sizeof(double), s));
    if (!c->hl.empty())
      CUDA_TRY(cudaMemcpyAsync(c->d_layers, c->hl.data(), c->hl.size() * sizeof(LayerDev),
                               cudaMemcpyHostToDevice, s));
    if (!c->hv.empty())
      CUDA_TRY(cudaMemcpyAsync(c->d_vecs, c->hv.data(), c->hv.size() * sizeof(VecDev), cudaMemcpyHostToDevice, s));
    for (int ph = 0; ph < kPhases; ++ph)
      if (!c->tiles[ph].empty())
        CUDA_TRY(cudaMemcpyAsync(c->d_tiles[ph], c->tiles[ph].data(), c->tiles[ph].size() * sizeof(Tile),
                                 cudaMemcpyHostToDevice, s));
    if (!c->pack.empty())
      CUDA_TRY(cudaMemcpyAsync(c->d_pack, c->pack.data(), c->pack.size() * sizeof(PackEntry),
                               cudaMemcpyHostToDevice, s));
    auto up = [&](void* dst, const void* src, size_t bytes) -> int {
      if (bytes) CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s));
      return PSGD_OK;
    };
    int rcu = up(c->d_gram_tiles, c->gram_tiles.data(), c->gram_tiles.size() * sizeof(Tile));
    if (!rcu) rcu = up(c->d_mat_u_tiles, c->mat_u_tiles.data(), c->mat_u_tiles.size() * sizeof(Tile));
    if (!rcu) rcu = up(c->d_xp, c->xp.data(), c->xp.size() * sizeof(XEntry));
    if (!rcu) rcu = up(c->d_xq, c->xq.data(), c->xq.size() * sizeof(XEntry));
    if (!rcu) rcu = up(c->d_ytiles, c->ytiles.data(), c->ytiles.size() * sizeof(Tile));
    if (rcu) return rcu;
    if (c->fused) {
      for (int q = 0; q < 2; ++q)
        if (!c->queue[q].empty())
          CUDA_TRY(cudaMemcpyAsync(c->d_queue[q], c->queue[q].data(), c->queue[q].size() * sizeof(Tile),
                                   cudaMemcpyHostToDevice, s));
      CUDA_TRY(cudaMemsetAsync(c->flags, 0, (size_t)c->n_flags * sizeof(unsigned), s));
    }
    CUDA_TRY(cudaMemsetAsync(c->sync_words, 0, 4 * sizeof(unsigned), s));
    if (!c->hl.empty()) {
      dim3 grid(64, (unsigned)c->hl.size());
      q_init_kernel<<<grid, 256, 0, s>>>(c->Qbar, c->d_layers, c->rank, c->rp, c->seed);
      CUDA_TRY(cudaGetLastError());
    }
    CUDA_TRY(cudaStreamSynchronize(s));
    if (rtopk) {
      int rc2 = rtopk_create(&c->rk, c->hl, c->hv, c->d_layers, c->d_vecs, c->W, c->seed, c->top_div, c->sample_div);
      if (rc2) return rc2;
    }
    return PSGD_OK;
  };
  rc = setup();
  if (rc) {
    cudaStreamSynchronize(c->stream);
    free_all(c);
    delete c;
    return rc;
  }
  *out = c;
  return PSGD_OK;
}

void psgd_destroy(psgd_ctx* c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  free_all(c);
  delete c;
}

int psgd_set_stream(psgd_ctx* c, void* cuda_stream) {
  if (!c) return fail(PSGD_ERR_INVALID, "context is NULL");
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  return PSGD_OK;
}

}  // extern "C"

namespace {

// One step; when X is not NULL the decompress phase also applies the
// momentum-SGD update to X and Mom.
// The kernel arguments of a step of context c (checked gradient pointers,
// the context's buffers); the caller sets the optional update fields.
int make_args(psgd_ctx* c, const float* const* grad_ptrs, float* out_update, StepArgs& a) {
  if (!grad_ptrs) return fail(PSGD_ERR_INVALID, "grad_ptrs must not be NULL");
  std::memset(&a, 0, sizeof(a));
  for (int w = 0; w < c->W; ++w) {
    if (!grad_ptrs[w]) return fail(PSGD_ERR_INVALID, "grad_ptrs[%d] is NULL", w);
    if (!aligned16(grad_ptrs[w])) return fail(PSGD_ERR_INVALID, "grad_ptrs[%d] is not 16-byte aligned", w);
    a.G[w] = grad_ptrs[w];
  }
  if (out_update && !aligned16(out_update)) return fail(PSGD_ERR_INVALID, "out_update is not 16-byte aligned");
  a.U = out_update;
  a.B = c->B;
  a.total = c->total;
  a.P = c->P;
  a.Phat = c->Phat;
  a.Qbar = c->Qbar;
  a.Qw = c->Qw;
  a.q_total = c->q_total;
  a.gram = c->gram;
  a.rinv = c->rinv;
  a.qpart = c->qpart;
  a.ppart = c->ppart;
  a.counters = c->counters;
  a.layers = c->d_layers;
  a.vecs = c->d_vecs;
  a.W = c->W;
  a.has_prev = c->has_prev;
  a.unbiased = c->unbiased ? 1 : 0;
  a.u_scale = 1.0f / ((float)c->W * (float)c->rank);
  a.stall_layer = -1;
  a.qbar_scale = 1.0f / (float)c->total_workers;
  a.sync = c->sync_words;
  return PSGD_OK;
}

int step_impl(psgd_ctx* c, const float* const* grad_ptrs, float* out_update, float* X, float* Mom, float lr,
              float beta) {
  const NvtxRange step_range("psgd step");
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (c->total_workers != c->W)
    return fail(PSGD_ERR_INVALID, "the workers of this context span processes: use psgd_step_begin/mid/end");
  StepArgs a;
  if ((rc = make_args(c, grad_ptrs, out_update, a))) return rc;
  a.X = X;
  a.Mom = Mom;
  a.lr = lr;
  a.beta = beta;
  // the decompress phase only writes U and the optional update
  const int phases = (out_update || X) ? kPhases : kPhases - 1;
  cudaEvent_t* ev = nullptr;
  if (c->timing) {
    ev = &c->ev[(size_t)(c->timed_since % kTimedSteps) * (kPhases + 1)];
    c->timed_since += 1;
    CUDA_TRY(cudaEventRecord(ev[0], c->stream));
  }
  if (c->rk) {
    if (X) return fail(PSGD_ERR_INVALID, "rTop-k has no fused momentum update");
    // phase slots: pass 0, pass 1, tail, apply (+ vectors)
    rc = rtopk_step(c->rk, grad_ptrs, c->B, c->total, out_update, c->steps, c->stream, ev ? ev + 1 : nullptr);
    if (rc) {
      c->broken = true;
      return rc;
    }
    c->has_prev = 1;
    c->steps += 1;
    return PSGD_OK;
  }
  if (c->unbiased && !c->hl.empty()) {
    // this step's Q: N(0,1) draws from the step's seed, shared by all workers
    dim3 grid(64, (unsigned)c->hl.size());
    q_init_kernel<<<grid, 256, 0, c->stream>>>(c->Qbar, c->d_layers, c->rank, c->rp, step_seed(c->seed, c->steps));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      c->broken = true;
      return cuda_fail(e, "Q draw launch");
    }
  }
  if (c->fused) {
    const int q = (out_update || X) ? 1 : 0;
    a.tiles = c->d_queue[q];
    a.n_items = (int32_t)c->queue[q].size();
    a.flags = c->flags;
    a.sync = c->sync_words;
    a.epoch = (uint32_t)(c->steps + 1);
    a.wait_ns = c->wait_ns;
    a.stall_layer = c->stall_layer;
    cudaError_t e = c->ks->launch_fused(a, std::min<int>(c->fused_ctas, a.n_items), c->stream);
    if (e != cudaSuccess) {
      c->broken = true;
      return cuda_fail(e, "fused step launch");
    }
    if (ev)
      for (int ph = 0; ph < kPhases; ++ph) CUDA_TRY(cudaEventRecord(ev[ph + 1], c->stream));
    c->has_prev = 1;
    c->steps += 1;
    return PSGD_OK;
  }
  if (c->ypath) {
    a.ypath = 1;
    a.ypart = c->ypart;
  }
  for (int ph = 0; ph < kPhases; ++ph) {
    const bool skip = c->unbiased && (ph == kOrthonormalise || ph == kBackProject);
    if (ph < phases && !skip) {
      const NvtxRange phase_range(kPhaseRange[ph]);
      a.tiles = c->d_tiles[ph];
      cudaError_t e;
      if (ph == kProject && c->ypath) {
        a.tiles = c->d_ytiles;
        a.y_clusters = c->y_clusters;
        e = c->ks->launch_cluster(a, c->y_clusters, kYClusterMax, c->y_smem, c->stream);
      } else if (ph == kBackProject && c->bmma) {
        e = c->ks->launch_bmma(a, (int)c->tiles[ph].size(), c->stream);
      } else {
        e = c->ks->launch(ph, a, (int)c->tiles[ph].size(), c->stream);
      }
      if (e != cudaSuccess) {
        c->broken = true;
        return cuda_fail(e, "phase kernel launch");
      }
    }
    if (ev) CUDA_TRY(cudaEventRecord(ev[ph + 1], c->stream));
  }
  c->has_prev = 1;
  c->steps += 1;
  return PSGD_OK;
}

}  // namespace

extern "C" {

int psgd_step(psgd_ctx* c, const float* const* grad_ptrs, float* out_update) {
  return step_impl(c, grad_ptrs, out_update, nullptr, nullptr, 0.f, 0.f);
}

int psgd_step_momentum(psgd_ctx* c, const float* const* grad_ptrs, float* params, float* momentum, float lr,
                       float beta, float* out_update) {
  if (!params || !momentum) return fail(PSGD_ERR_INVALID, "params and momentum must not be NULL");
  if (!aligned16(params) || !aligned16(momentum))
    return fail(PSGD_ERR_INVALID, "params and momentum must be 16-byte aligned");
  if (!std::isfinite(lr) || !std::isfinite(beta)) return fail(PSGD_ERR_INVALID, "lr and beta must be finite");
  return step_impl(c, grad_ptrs, out_update, params, momentum, lr, beta);
}

int psgd_exchange_sizes(const psgd_ctx* c, int64_t* p_floats, int64_t* q_floats) {
  if (!c) return fail(PSGD_ERR_INVALID, "context is NULL");
  if (p_floats) *p_floats = c->xp_floats;
  if (q_floats) *q_floats = c->xq_floats;
  return PSGD_OK;
}

}  // extern "C"

namespace {

int split_ok(psgd_ctx* c, int phase, const char* what) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (c->rk || c->unbiased) return fail(PSGD_ERR_INVALID, "%s: the split step is for PowerSGD contexts", what);
  if (c->split_phase != phase)
    return fail(PSGD_ERR_INVALID, "%s called out of order (begin, mid, end)", what);
  return PSGD_OK;
}

int xchg(psgd_ctx* c, const StepArgs& a, float* dense, float* padded, const std::vector<XEntry>& ent,
         const XEntry* d_ent, int to_dense) {
  if (ent.empty()) return PSGD_OK;
  dim3 grid(16, (unsigned)ent.size());
  xchg_kernel<<<grid, 256, 0, c->stream>>>(a, dense, padded, d_ent, c->rank, c->rp, to_dense);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    c->broken = true;
    return cuda_fail(e, "exchange kernel");
  }
  return PSGD_OK;
}

int launch_phase(psgd_ctx* c, int phase, StepArgs& a, const Tile* tiles, int n) {
  a.tiles = tiles;
  cudaError_t e = (phase < 0)                           ? c->ks->launch_gram(a, n, c->stream)
                  : (phase == kBackProject && c->bmma) ? c->ks->launch_bmma(a, n, c->stream)
                                                        : c->ks->launch(phase, a, n, c->stream);
  if (e != cudaSuccess) {
    c->broken = true;
    return cuda_fail(e, "phase kernel launch");
  }
  return PSGD_OK;
}

}  // namespace

extern "C" {

int psgd_step_begin(psgd_ctx* c, const float* const* grad_ptrs, float* p_out) {
  int rc = split_ok(c, 0, "psgd_step_begin");
  if (rc) return rc;
  if (!p_out && c->xp_floats) return fail(PSGD_ERR_INVALID, "p_out must not be NULL");
  StepArgs a;
  if ((rc = make_args(c, grad_ptrs, nullptr, a))) return rc;
  a.split = 1;
  if ((rc = launch_phase(c, kProject, a, c->d_tiles[kProject], (int)c->tiles[kProject].size()))) return rc;
  if ((rc = xchg(c, a, p_out, c->P, c->xp, c->d_xp, 1))) return rc;
  c->split_grads.assign(grad_ptrs, grad_ptrs + c->W);
  c->split_phase = 1;
  return PSGD_OK;
}

int psgd_step_mid(psgd_ctx* c, const float* p_sum, float* q_out) {
  int rc = split_ok(c, 1, "psgd_step_mid");
  if (rc) return rc;
  if ((!p_sum && c->xp_floats) || (!q_out && c->xq_floats))
    return fail(PSGD_ERR_INVALID, "p_sum and q_out must not be NULL");
  StepArgs a;
  if ((rc = make_args(c, c->split_grads.data(), nullptr, a))) return rc;
  if ((rc = xchg(c, a, const_cast<float*>(p_sum), c->P, c->xp, c->d_xp, 0))) return rc;
  if ((rc = launch_phase(c, -1, a, c->d_gram_tiles, (int)c->gram_tiles.size()))) return rc;
  if ((rc = launch_phase(c, kOrthonormalise, a, c->d_tiles[kOrthonormalise], (int)c->tiles[kOrthonormalise].size())))
    return rc;
  if ((rc = launch_phase(c, kBackProject, a, c->d_tiles[kBackProject], (int)c->tiles[kBackProject].size())))
    return rc;
  if ((rc = xchg(c, a, q_out, c->Qbar, c->xq, c->d_xq, 1))) return rc;
  c->split_phase = 2;
  return PSGD_OK;
}

int psgd_step_end(psgd_ctx* c, const float* q_sum, float* out_update) {
  int rc = split_ok(c, 2, "psgd_step_end");
  if (rc) return rc;
  if (!q_sum && c->xq_floats) return fail(PSGD_ERR_INVALID, "q_sum must not be NULL");
  StepArgs a;
  if ((rc = make_args(c, c->split_grads.data(), out_update, a))) return rc;
  if ((rc = xchg(c, a, const_cast<float*>(q_sum), c->Qbar, c->xq, c->d_xq, 0))) return rc;
  if (out_update &&
      (rc = launch_phase(c, kDecompress, a, c->d_mat_u_tiles, (int)c->mat_u_tiles.size())))
    return rc;
  c->split_phase = 0;
  c->has_prev = 1;
  c->steps += 1;
  return PSGD_OK;
}

int psgd_sync(psgd_ctx* c) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  return sync_and_check(c);
}

int psgd_set_timing(psgd_ctx* c, int on) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (on && c->ev.empty()) {
    c->ev.assign((size_t)kTimedSteps * (kPhases + 1), nullptr);
    for (auto& e : c->ev) CUDA_TRY(cudaEventCreate(&e));
  }
  c->timing = on != 0;
  c->timed_since = 0;
  return PSGD_OK;
}

int psgd_get_phase_times(psgd_ctx* c, float* ms) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (!ms) return fail(PSGD_ERR_INVALID, "ms must not be NULL");
  if (!c->timing) return fail(PSGD_ERR_INVALID, "phase timing is off (psgd_options.timing)");
  if (c->timed_since == 0) return fail(PSGD_ERR_INVALID, "no step since the last call");
  if ((rc = sync_and_check(c))) return rc;
  const int64_t nsteps = std::min<int64_t>(c->timed_since, kTimedSteps);
  const int64_t first = c->timed_since - nsteps;
  for (int ph = 0; ph < kPhases; ++ph) ms[ph] = 0.f;
  for (int64_t t = first; t < c->timed_since; ++t) {
    const cudaEvent_t* ev = &c->ev[(size_t)(t % kTimedSteps) * (kPhases + 1)];
    for (int ph = 0; ph < kPhases; ++ph) {
      float x = 0.f;
      CUDA_TRY(cudaEventElapsedTime(&x, ev[ph], ev[ph + 1]));
      ms[ph] += x;
    }
  }
  for (int ph = 0; ph < kPhases; ++ph) ms[ph] /= (float)nsteps;
  c->timed_since = 0;
  return PSGD_OK;
}

int psgd_step_host(psgd_ctx* c, const float* const* grad_host, float* msg_host, float* update_host) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (!grad_host || !msg_host) return fail(PSGD_ERR_INVALID, "grad_host and msg_host must not be NULL");
  const int W = c->W;
  if (!c->stage_U) {
    rc = dalloc(&c->stage_U, c->total, "stage_U");
    if (!rc) rc = dalloc(&c->stage_msg, c->msg_floats, "stage_msg");
    if (rc) return rc;
  }
  // A pinned, mapped host buffer is read in place by the kernels over the
  // CPU-GPU link (its device alias); any other buffer is copied to staging.
  std::vector<const float*> dptr(W);
  for (int w = 0; w < W; ++w) {
    if (!grad_host[w]) return fail(PSGD_ERR_INVALID, "grad_host[%d] is NULL", w);
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, grad_host[w]) != cudaSuccess) {
      cudaGetLastError();
      at.type = cudaMemoryTypeUnregistered;
    }
    if (at.type == cudaMemoryTypeHost && at.devicePointer && aligned16(at.devicePointer)) {
      dptr[w] = static_cast<const float*>(at.devicePointer);
      continue;
    }
    if (!c->stage_G && (rc = dalloc(&c->stage_G, (int64_t)W * c->total, "stage_G"))) return rc;
    dptr[w] = c->stage_G + (int64_t)w * c->total;
    CUDA_TRY(cudaMemcpyAsync(const_cast<float*>(dptr[w]), grad_host[w], (size_t)c->total * sizeof(float),
                             cudaMemcpyHostToDevice, c->stream));
  }
  rc = psgd_step(c, dptr.data(), update_host ? c->stage_U : nullptr);
  if (rc) return rc;
  if (c->rk) {  // per matrix layer and worker: k indices, then k values; gathered, then one copy
    if ((rc = rtopk_pack(c->rk, c->stage_msg, c->stream))) return rc;
    if (c->msg_floats)
      CUDA_TRY(cudaMemcpyAsync(msg_host, c->stage_msg, (size_t)c->msg_floats * sizeof(float),
                               cudaMemcpyDeviceToHost, c->stream));
  } else if (!c->pack.empty()) {
    dim3 grid(32, (unsigned)c->pack.size());
    pack_msg_kernel<<<grid, 256, 0, c->stream>>>(c->stage_msg, c->unbiased ? c->P : c->Phat, c->Qbar, c->d_pack,
                                                 c->rank, c->rp);
    CUDA_TRY(cudaGetLastError());
    CUDA_TRY(cudaMemcpyAsync(msg_host, c->stage_msg, (size_t)c->msg_floats * sizeof(float),
                             cudaMemcpyDeviceToHost, c->stream));
  }
  if (update_host)
    CUDA_TRY(cudaMemcpyAsync(update_host, c->stage_U, (size_t)c->total * sizeof(float), cudaMemcpyDeviceToHost,
                             c->stream));
  return sync_and_check(c);
}

int psgd_get_PQ(psgd_ctx* c, int layer, float* P, float* Q) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (c->rk) return fail(PSGD_ERR_INVALID, "rTop-k keeps no factors");
  const LayerDev* L;
  if ((rc = matrix_layer(c, layer, &L))) return rc;
  const size_t rb = (size_t)c->rank * sizeof(float), pb = (size_t)c->rp * sizeof(float);
  if (P) CUDA_TRY(cudaMemcpy2DAsync(P, rb, (c->unbiased ? c->P : c->Phat) + L->p_off, pb, rb, L->n, cudaMemcpyDefault, c->stream));
  if (Q) CUDA_TRY(cudaMemcpy2DAsync(Q, rb, c->Qbar + L->q_off, pb, rb, L->m, cudaMemcpyDefault, c->stream));
  return sync_and_check(c);
}

int psgd_get_sparse(psgd_ctx* c, int layer, int worker, int32_t* idx, float* val, int64_t* count) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (!c->rk) return fail(PSGD_ERR_INVALID, "not an rTop-k context");
  const LayerDev* L;
  if ((rc = matrix_layer(c, layer, &L))) return rc;
  if (worker < 0 || worker >= c->W) return fail(PSGD_ERR_INVALID, "worker %d out of range", worker);
  const int mi = c->mat_of[layer];
  const int64_t k = rtopk_k(c->rk, mi);
  const int32_t* di;
  const float* dv;
  rtopk_message(c->rk, mi, worker, &di, &dv);
  if (count) *count = k;
  if (idx) CUDA_TRY(cudaMemcpyAsync(idx, di, (size_t)k * sizeof(int32_t), cudaMemcpyDefault, c->stream));
  if (val) CUDA_TRY(cudaMemcpyAsync(val, dv, (size_t)k * sizeof(float), cudaMemcpyDefault, c->stream));
  return sync_and_check(c);
}

int psgd_get_Qw(psgd_ctx* c, int layer, int worker, float* Q) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  const LayerDev* L;
  if ((rc = matrix_layer(c, layer, &L))) return rc;
  if (worker < 0 || worker >= c->W) return fail(PSGD_ERR_INVALID, "worker %d out of range", worker);
  if (!Q) return fail(PSGD_ERR_INVALID, "Q must not be NULL");
  if (c->unbiased || c->rk) return fail(PSGD_ERR_INVALID, "this compressor forms no Q_w");
  const size_t rb = (size_t)c->rank * sizeof(float), pb = (size_t)c->rp * sizeof(float);
  CUDA_TRY(cudaMemcpy2DAsync(Q, rb, c->Qw + (int64_t)worker * c->q_total + L->q_off, pb, rb, L->m,
                             cudaMemcpyDefault, c->stream));
  return sync_and_check(c);
}

int psgd_get_error(psgd_ctx* c, int layer, int worker, float* E) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  const LayerDev* L;
  if ((rc = matrix_layer(c, layer, &L))) return rc;
  if (worker < 0 || worker >= c->W) return fail(PSGD_ERR_INVALID, "worker %d out of range", worker);
  if (!E) return fail(PSGD_ERR_INVALID, "E must not be NULL");
  const int64_t nm = (int64_t)L->n * L->m;
  float* dst = E;
  const bool dev = is_device_ptr(E);
  if (c->unbiased) {  // no error feedback: the error is zero
    if (dev) {
      CUDA_TRY(cudaMemsetAsync(E, 0, (size_t)nm * sizeof(float), c->stream));
      return sync_and_check(c);
    }
    std::memset(E, 0, (size_t)nm * sizeof(float));
    return PSGD_OK;
  }
  if (!dev) {
    if (c->e_scratch_elems < nm) {
      if (c->e_scratch) cudaFree(c->e_scratch);
      c->e_scratch = nullptr;
      c->e_scratch_elems = 0;
      if ((rc = dalloc(&c->e_scratch, nm, "error scratch"))) return rc;
      c->e_scratch_elems = nm;
    }
    dst = c->e_scratch;
  }
  const float* Bw = c->B + (int64_t)worker * c->total + L->off;
  const float* Qw = c->Qw + (int64_t)worker * c->q_total + L->q_off;
  CUDA_TRY(c->ks->error(dst, Bw, c->Phat + L->p_off, Qw, L->n, L->m, L->ld, c->stream));
  if (!dev) CUDA_TRY(cudaMemcpyAsync(E, dst, (size_t)nm * sizeof(float), cudaMemcpyDeviceToHost, c->stream));
  return sync_and_check(c);
}

int psgd_set_state(psgd_ctx* c, int layer, const float* Q, const float* const* E) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  const LayerDev* L;
  if ((rc = matrix_layer(c, layer, &L))) return rc;
  if (!Q) return fail(PSGD_ERR_INVALID, "Q must not be NULL");
  if (c->unbiased || c->rk) return fail(PSGD_ERR_INVALID, "this compressor's state cannot be set");
  if (E)
    for (int w = 0; w < c->W; ++w)
      if (!E[w]) return fail(PSGD_ERR_INVALID, "E[%d] is NULL", w);
  cudaStream_t s = c->stream;
  const size_t rb = (size_t)c->rank * sizeof(float), pb = (size_t)c->rp * sizeof(float);
  CUDA_TRY(cudaMemsetAsync(c->Qbar + L->q_off, 0, (size_t)L->ld * c->rp * sizeof(float), s));
  CUDA_TRY(cudaMemcpy2DAsync(c->Qbar + L->q_off, pb, Q, rb, rb, L->m, cudaMemcpyDefault, s));
  CUDA_TRY(cudaMemsetAsync(c->Phat + L->p_off, 0, (size_t)L->n * c->rp * sizeof(float), s));
  for (int w = 0; w < c->W; ++w) {
    float* Bw = c->B + (int64_t)w * c->total + L->off;
    CUDA_TRY(cudaMemsetAsync(c->Qw + (int64_t)w * c->q_total + L->q_off, 0, (size_t)L->ld * c->rp * sizeof(float), s));
    CUDA_TRY(cudaMemsetAsync(Bw, 0, (size_t)L->n * L->ld * sizeof(float), s));
    if (E)
      CUDA_TRY(cudaMemcpy2DAsync(Bw, (size_t)L->ld * sizeof(float), E[w], (size_t)L->m * sizeof(float),
                                 (size_t)L->m * sizeof(float), L->n, cudaMemcpyDefault, s));
  }
  return sync_and_check(c);
}

int psgd_get_stats(const psgd_ctx* c, psgd_stats* out) {
  if (!c || !out) return fail(PSGD_ERR_INVALID, "NULL argument");
  std::memset(out, 0, sizeof(*out));
  out->steps = c->steps;
  out->floats_sent_per_step = c->sent_step;
  out->floats_uncompressed_per_step = c->unc_step;
  out->floats_sent = c->sent_step * c->steps;
  out->floats_uncompressed = c->unc_step * c->steps;
  out->matrix_elements = c->mat_el;
  out->vector_elements = c->vec_el;
  out->buffer_elements = c->total;
  for (int ph = 0; ph < kPhases; ++ph) out->tiles[ph] = (int64_t)c->tiles[ph].size();
  if (c->ypath) out->tiles[kProject] = (int64_t)c->y_clusters * kYClusterMax;
  out->one_pass_project = c->ypath ? 1 : 0;
  out->kernel_rank = c->rp;
  for (int i = 0; i < 3; ++i) out->tile_rows[i] = c->tile_rows[i];
  out->launches_per_step = kPhases + (c->rp >= 8 ? 1 : 0);  // r >= 8: the second pass's Phat rows
  // the unbiased variant: Q draw, project, decompress
  if (c->unbiased) out->launches_per_step = 3;
  if (c->fused) out->launches_per_step = 1;
  out->fused_step = c->fused ? 1 : 0;
  if (c->rk) out->launches_per_step = rtopk_launches(c->rk);
  out->message_floats = c->msg_floats;
  return PSGD_OK;
}

int psgd_layer_flags(psgd_ctx* c, int layer, int32_t* flags) {
  int rc = ctx_ok(c);
  if (rc) return rc;
  if (!flags) return fail(PSGD_ERR_INVALID, "flags must not be NULL");
  const LayerDev* L = nullptr;
  if ((rc = matrix_layer(c, layer, &L))) return rc;
  *flags = 0;
  if (c->steps == 0) return PSGD_OK;
  double f[2] = {0.0, 0.0};
  const int64_t at = L->rinv_off + 2 * (int64_t)c->rp * c->rp + c->rp;
  CUDA_TRY(cudaMemcpyAsync(f, c->rinv + at, sizeof(f), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  *flags = (f[0] != 0.0 ? 1 : 0) | (f[1] != 0.0 ? 2 : 0);
  return PSGD_OK;
}

int psgd_layer_info(const psgd_ctx* c, int layer, int64_t* offset, int64_t* n, int64_t* m, int64_t* ld) {
  if (!c) return fail(PSGD_ERR_INVALID, "context is NULL");
  if (layer < 0 || layer >= c->num_layers) return fail(PSGD_ERR_INVALID, "layer %d out of range", layer);
  if (offset) *offset = c->off[layer];
  if (n) *n = c->n[layer];
  if (m) *m = c->m[layer];
  if (ld) *ld = c->ld[layer];
  return PSGD_OK;
}

}  // extern "C"
