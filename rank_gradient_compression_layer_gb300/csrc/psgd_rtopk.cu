// rTop-k sparsification (rTop-k review page, "rTop-k: A Statistical
// Estimation Approach to Distributed SGD", proposed method, bullet 3: a
// random subset of the top-k magnitude entries), with error feedback.
//
// Per (worker w, matrix layer l) problem, over the layer's d entries in
// row-major order (flat index i):
//   M = G + E (float32, written back into E's buffer B)
//   top set T: the r entries with the largest (|M|, -i)   r = ceil(d / top_div)
//   sent set K: the k members of T with the smallest (h(i), i)
//               k = ceil(r / sample_div), h(i) the upper 32 bits of
//               splitmix64(key(seed, step, w, l) + (i + 1) gamma)
//   E <- M with K zeroed; the message is K's indices (ascending) and values
//   U = (sum_w S_w) / W, summed in worker order (float32)
//
// Both selections are radix selects over composite 64-bit keys that are
// unique per entry -- (|M| bits, ~i) and (h(i), i) -- so the k-th key is one
// value and "key >= / <= threshold" selects exactly r / k entries.  Six
// 11-bit digit passes per select; each pass histograms the digit of the
// entries still matching the prefix found so far, and the last CTA of a
// problem to finish its chunk picks the digit and narrows the prefix.  A
// count / scan / apply sequence then writes every worker's message in index
// order and U, so the whole step is deterministic.
#include <cuda_runtime.h>

#include <cstring>
#include <vector>

#include "psgd_kernels.cuh"
#include "psgd_plan.h"
#include "psgd_rtopk.h"

namespace psgd {
namespace {

constexpr int kRkThreads = 256;
constexpr int kRkPer = 8;                        // consecutive entries per thread
constexpr int kRkChunk = kRkThreads * kRkPer;    // entries per tile
constexpr int kRkBins = 2048;                    // 11-bit digits
constexpr int kRkPasses = 6;
__constant__ int c_shift[kRkPasses] = {53, 42, 31, 20, 9, 0};
__constant__ int c_width[kRkPasses] = {11, 11, 11, 11, 11, 9};
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

struct RkProb {   // one (worker, matrix layer) problem
  int32_t mi, w;  // matrix layer position, worker
  int64_t d, r, k;
  int64_t nchunks, chunk0;  // chunks of the layer; first chunk counter of this problem
  int64_t msg_off;          // first message entry of this problem
};

struct RkState {
  uint64_t prefix;  // key bits found so far (bits above the current digit)
  int64_t need;     // entries still to take from those matching the prefix
  uint64_t vm;      // magnitude threshold: T = {Km >= vm}
  uint64_t vr;      // draw threshold: K = {i in T : Kr <= vr}
  uint64_t dkey;    // draw stream key of this step
  int32_t done;     // the current select needs no further digits
  int32_t pad;
};

struct RkTile {
  int32_t p;      // problem (hist passes) or matrix layer (count / apply)
  int32_t chunk;
};

struct RkArgs {
  const float* G[kMaxWorkers];
  float* B;
  float* U;
  int64_t total;
  const LayerDev* layers;
  const RkProb* probs;
  RkState* state;
  uint32_t* hist;     // problems x kRkBins
  unsigned* arrive;   // problems
  const RkTile* tiles;
  int64_t* ccount;    // per problem chunk counts, then exclusive offsets
  int32_t* sidx;
  float* sval;
  int32_t W, nmat;
  uint64_t seed;
  int64_t step;
};

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t key_mag(float m, int64_t i) {
  const uint32_t pat = __float_as_uint(m) & 0x7FFFFFFFu;
  return ((uint64_t)pat << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
}

__device__ __forceinline__ uint64_t key_draw(uint64_t dkey, int64_t i) {
  const uint64_t h = mix64(dkey + (uint64_t)(i + 1) * kGamma) >> 32;
  return (h << 32) | (uint64_t)(uint32_t)i;
}

// Packed-buffer position of flat entry i of layer L.
__device__ __forceinline__ int64_t pos_of(const LayerDev& L, int64_t i) {
  const int64_t row = i / L.m;
  return L.off + row * L.ld + (i - row * L.m);
}

// Last CTA of a problem's pass: pick the digit at `shift` of the need-th key
// (largest first for the top set, smallest first for the draw) and narrow
// the prefix.  h: the pass's histogram in shared memory.
__device__ void rk_find(RkState& st, const uint32_t* h, int shift, int width, bool largest, uint64_t* s_sum) {
  const int t = threadIdx.x;
  const int nb = 1 << width;
  const int per = kRkBins / kRkThreads;  // 8 bins per thread
  // thread t owns walk positions [t per, t per + per); walk position j is
  // bin nb - 1 - j (largest first) or bin j (smallest first)
  uint64_t mine = 0;
  for (int j = t * per; j < t * per + per; ++j)
    if (j < nb) mine += h[largest ? nb - 1 - j : j];
  s_sum[t] = mine;
  __syncthreads();
  // inclusive scan over threads (Hillis-Steele)
  for (int o = 1; o < kRkThreads; o <<= 1) {
    const uint64_t v = (t >= o) ? s_sum[t - o] : 0;
    __syncthreads();
    s_sum[t] += v;
    __syncthreads();
  }
  const uint64_t incl = s_sum[t], excl = incl - mine, all = s_sum[kRkThreads - 1];
  const uint64_t mask_above = (shift + width >= 64) ? 0ull : (~0ull << (shift + width));
  if (t == 0 && (uint64_t)st.need > all) {
    // every entry matching the prefix is taken: the threshold is the lowest
    // (largest first) or highest (smallest first) key with that prefix
    st.prefix = largest ? (st.prefix & mask_above) : ((st.prefix & mask_above) | ~mask_above);
    st.done = 1;
  }
  __syncthreads();
  if (st.done) return;
  if (excl < (uint64_t)st.need && (uint64_t)st.need <= incl) {
    uint64_t c = excl;
    for (int j = t * per; j < t * per + per && j < nb; ++j) {
      const int b = largest ? nb - 1 - j : j;
      if (c + h[b] >= (uint64_t)st.need) {
        st.prefix = (st.prefix & mask_above) | ((uint64_t)b << shift);
        st.need -= (int64_t)c;
        break;
      }
      c += h[b];
    }
  }
}

// One digit pass of one select over all problems.  draw = false: the top
// set by magnitude (pass 0 also forms M = G + E into B); draw = true: the
// sent subset among the top set.
__global__ void __launch_bounds__(kRkThreads) rk_hist_kernel(RkArgs a, int q, int draw) {
  __shared__ uint32_t h[kRkBins];
  __shared__ uint64_t s_sum[kRkThreads];
  __shared__ int s_flag;
  const RkTile t = a.tiles[blockIdx.x];
  const RkProb P = a.probs[t.p];
  const LayerDev L = a.layers[P.mi];
  RkState* stp = a.state + t.p;
  const int shift = c_shift[q], width = c_width[q];
  const uint64_t mask_above = (shift + width >= 64) ? 0ull : (~0ull << (shift + width));
  const uint64_t prefix = stp->prefix, vm = stp->vm, dkey = stp->dkey;
  const bool skip = stp->done != 0;
  for (int b = threadIdx.x; b < kRkBins; b += blockDim.x) h[b] = 0u;
  __syncthreads();
  if (!skip) {
    const int64_t i0 = (int64_t)t.chunk * kRkChunk + (int64_t)threadIdx.x * kRkPer;
    float* Bw = a.B + (int64_t)P.w * a.total;
    const float* Gw = a.G[P.w];
    for (int j = 0; j < kRkPer; ++j) {
      const int64_t i = i0 + j;
      if (i >= P.d) break;
      const int64_t pos = pos_of(L, i);
      float m;
      if (!draw && q == 0) {
        m = __ldcs(Gw + pos) + Bw[pos];
        Bw[pos] = m;
      } else {
        m = Bw[pos];
      }
      uint64_t K = key_mag(m, i);
      if (draw) {
        if (K < vm) continue;  // not in the top set
        K = key_draw(dkey, i);
      }
      if ((K & mask_above) == (prefix & mask_above)) atomicAdd(&h[(K >> shift) & (uint64_t)((1 << width) - 1)], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = a.hist + (int64_t)t.p * kRkBins;
  if (!skip)
    for (int b = threadIdx.x; b < kRkBins; b += blockDim.x)
      if (h[b]) atomicAdd(gh + b, h[b]);
  if (!cta_arrive_last(a.arrive + t.p, (unsigned)P.nchunks, &s_flag)) return;
  // last CTA of the problem: the digit, then a clean histogram for the next pass
  for (int b = threadIdx.x; b < kRkBins; b += blockDim.x) {
    h[b] = __ldcg(gh + b);
    gh[b] = 0u;
  }
  __syncthreads();
  __shared__ RkState s_st;
  if (threadIdx.x == 0) s_st = *stp;
  __syncthreads();
  if (!s_st.done) rk_find(s_st, h, shift, width, !draw, s_sum);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (q == kRkPasses - 1) {
      if (!draw) {  // the top set is fixed: start the draw select
        s_st.vm = s_st.prefix;
        s_st.prefix = 0;
        s_st.need = P.k;
        s_st.done = 0;
      } else {
        s_st.vr = s_st.prefix;
      }
    }
    *stp = s_st;
  }
}

// Sent entries of layer mi per chunk and worker (for the index-ordered
// message offsets).  Thread = 8 consecutive entries.
__global__ void __launch_bounds__(kRkThreads) rk_count_kernel(RkArgs a) {
  __shared__ int s_part[kRkThreads / 32];
  const RkTile t = a.tiles[blockIdx.x];
  const int mi = t.p;
  const LayerDev L = a.layers[mi];
  const int64_t i0 = (int64_t)t.chunk * kRkChunk + (int64_t)threadIdx.x * kRkPer;
  for (int w = 0; w < a.W; ++w) {
    const int p = w * a.nmat + mi;
    const RkProb P = a.probs[p];
    const RkState st = a.state[p];
    const float* Bw = a.B + (int64_t)w * a.total;
    int c = 0;
    for (int j = 0; j < kRkPer; ++j) {
      const int64_t i = i0 + j;
      if (i >= P.d) break;
      const float m = Bw[pos_of(L, i)];
      if (key_mag(m, i) >= st.vm && key_draw(st.dkey, i) <= st.vr) ++c;
    }
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = 0;
      for (int v = 0; v < kRkThreads / 32; ++v) s += s_part[v];
      a.ccount[P.chunk0 + t.chunk] = s;
    }
    __syncthreads();
  }
}

// Exclusive offsets of each problem's chunk counts (one CTA per problem).
__global__ void __launch_bounds__(kRkThreads) rk_scan_kernel(RkArgs a) {
  __shared__ int64_t s_sum[kRkThreads];
  const RkProb P = a.probs[blockIdx.x];
  int64_t* c = a.ccount + P.chunk0;
  const int64_t per = (P.nchunks + kRkThreads - 1) / kRkThreads;
  const int64_t b0 = threadIdx.x * per, b1 = min(P.nchunks, b0 + per);
  int64_t mine = 0;
  for (int64_t b = b0; b < b1; ++b) mine += c[b];
  s_sum[threadIdx.x] = mine;
  __syncthreads();
  for (int o = 1; o < kRkThreads; o <<= 1) {
    const int64_t v = (threadIdx.x >= (unsigned)o) ? s_sum[threadIdx.x - o] : 0;
    __syncthreads();
    s_sum[threadIdx.x] += v;
    __syncthreads();
  }
  int64_t run = s_sum[threadIdx.x] - mine;
  for (int64_t b = b0; b < b1; ++b) {
    const int64_t x = c[b];
    c[b] = run;
    run += x;
  }
}

// Messages, error and update of layer mi over one chunk, all workers in
// order: the sent entries go to the worker's message at their index-ordered
// position, are zeroed in B (E = M - S), and summed into U.
__global__ void __launch_bounds__(kRkThreads) rk_apply_kernel(RkArgs a) {
  __shared__ int s_warp[kRkThreads / 32];
  const RkTile t = a.tiles[blockIdx.x];
  const int mi = t.p;
  const LayerDev L = a.layers[mi];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i0 = (int64_t)t.chunk * kRkChunk + (int64_t)threadIdx.x * kRkPer;
  float u[kRkPer];
#pragma unroll
  for (int j = 0; j < kRkPer; ++j) u[j] = 0.f;
  for (int w = 0; w < a.W; ++w) {
    const int p = w * a.nmat + mi;
    const RkProb P = a.probs[p];
    const RkState st = a.state[p];
    float* Bw = a.B + (int64_t)w * a.total;
    bool sel[kRkPer];
    float mv[kRkPer];
    int c = 0;
#pragma unroll
    for (int j = 0; j < kRkPer; ++j) {
      const int64_t i = i0 + j;
      sel[j] = false;
      mv[j] = 0.f;
      if (i < P.d) {
        mv[j] = Bw[pos_of(L, i)];
        sel[j] = key_mag(mv[j], i) >= st.vm && key_draw(st.dkey, i) <= st.vr;
        c += sel[j] ? 1 : 0;
      }
    }
    // exclusive rank of this thread's first sent entry within the chunk
    int incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int v = 0; v < warp; ++v) base += s_warp[v];
    __syncthreads();
    int64_t at = P.msg_off + a.ccount[P.chunk0 + t.chunk] + base + incl - c;
    const int64_t end = P.msg_off + P.k;  // exactly k entries are selected; never write past them
#pragma unroll
    for (int j = 0; j < kRkPer; ++j) {
      if (sel[j]) {
        const int64_t i = i0 + j;
        if (at < end) {
          a.sidx[at] = (int32_t)i;
          a.sval[at] = mv[j];
        }
        ++at;
        u[j] += mv[j];
        Bw[pos_of(L, i)] = 0.f;
      }
    }
  }
  if (a.U) {
    const float inv = 1.0f / (float)a.W;
#pragma unroll
    for (int j = 0; j < kRkPer; ++j) {
      const int64_t i = i0 + j;
      if (i < (int64_t)L.n * L.m) a.U[pos_of(L, i)] = u[j] * inv;
    }
  }
}

// Vector layers: U = the worker mean (one thread per entry).
__global__ void rk_vec_kernel(const VecDev* vecs, int nvec, RkArgs a) {
  for (int vi = 0; vi < nvec; ++vi) {
    const VecDev V = vecs[vi];
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < V.n; i += (int64_t)gridDim.x * blockDim.x) {
      float s = 0.f;
      for (int w = 0; w < a.W; ++w) s += a.G[w][V.off + i];
      a.U[V.off + i] = s / (float)a.W;
    }
  }
}

// Per-step draw keys and select state of every problem.
__global__ void rk_begin_kernel(RkArgs a, int nprob) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= nprob) return;
  const RkProb P = a.probs[p];
  const LayerDev L = a.layers[P.mi];
  const uint64_t s = mix64(a.seed + (uint64_t)(a.step + 1) * kGamma);
  RkState st;
  st.prefix = 0;
  st.need = P.r;
  st.vm = 0;
  st.vr = 0;
  st.dkey = mix64(s + (uint64_t)(P.w * 65536 + L.index + 1) * kGamma);
  st.done = 0;
  st.pad = 0;
  a.state[p] = st;
}

}  // namespace

struct RTopK {
  int W = 0, nmat = 0, nprob = 0;
  uint64_t seed = 0;
  std::vector<RkProb> hp;
  std::vector<int64_t> kk;  // k per matrix layer
  std::vector<RkTile> htiles, ltiles;
  const LayerDev* d_layers = nullptr;
  const VecDev* d_vecs = nullptr;
  int nvec = 0;
  RkProb* d_probs = nullptr;
  RkState* d_state = nullptr;
  uint32_t* d_hist = nullptr;
  unsigned* d_arrive = nullptr;
  RkTile* d_htiles = nullptr;
  RkTile* d_ltiles = nullptr;
  int64_t* d_ccount = nullptr;
  int32_t* d_sidx = nullptr;
  float* d_sval = nullptr;
  int64_t nchunk_total = 0, msg_total = 0;
};

namespace {

template <class T>
int rk_alloc(T** p, int64_t count, const char* what) {
  if (count <= 0) count = 1;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), (size_t)count * sizeof(T));
  if (e != cudaSuccess) {
    *p = nullptr;
    return cuda_fail(e, what);
  }
  return PSGD_OK;
}

}  // namespace

void rtopk_destroy(RTopK* rk) {
  if (!rk) return;
  void* ptrs[] = {rk->d_probs, rk->d_state, rk->d_hist, rk->d_arrive, rk->d_htiles, rk->d_ltiles,
                  rk->d_ccount, rk->d_sidx, rk->d_sval};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  delete rk;
}

int rtopk_create(RTopK** out, const std::vector<LayerDev>& hl, const std::vector<VecDev>& hv,
                 const LayerDev* d_layers, const VecDev* d_vecs, int W, uint64_t seed, int top_div,
                 int sample_div) {
  *out = nullptr;
  if (top_div < 1 || sample_div < 1) return fail(PSGD_ERR_INVALID, "rTop-k divisors must be >= 1");
  RTopK* rk = new RTopK();
  rk->W = W;
  rk->nmat = (int)hl.size();
  rk->nprob = W * rk->nmat;
  rk->seed = seed;
  rk->d_layers = d_layers;
  rk->d_vecs = d_vecs;
  rk->nvec = (int)hv.size();
  for (int mi = 0; mi < rk->nmat; ++mi) {
    const int64_t d = (int64_t)hl[mi].n * hl[mi].m;
    if (d >= ((int64_t)1 << 31)) {
      delete rk;
      return fail(PSGD_ERR_INVALID, "rTop-k needs layers of fewer than 2^31 entries");
    }
    const int64_t r = ceil_div(d, top_div);
    rk->kk.push_back(ceil_div(r, sample_div));
  }
  for (int w = 0; w < W; ++w)
    for (int mi = 0; mi < rk->nmat; ++mi) {
      const int64_t d = (int64_t)hl[mi].n * hl[mi].m;
      RkProb P;
      P.mi = mi;
      P.w = w;
      P.d = d;
      P.r = ceil_div(d, top_div);
      P.k = rk->kk[mi];
      P.nchunks = ceil_div(d, kRkChunk);
      P.chunk0 = rk->nchunk_total;
      rk->nchunk_total += P.nchunks;
      P.msg_off = rk->msg_total;
      rk->msg_total += P.k;
      rk->hp.push_back(P);
      for (int64_t c = 0; c < P.nchunks; ++c) rk->htiles.push_back({(int32_t)(w * rk->nmat + mi), (int32_t)c});
    }
  for (int mi = 0; mi < rk->nmat; ++mi)
    for (int64_t c = 0; c < rk->hp[mi].nchunks; ++c) rk->ltiles.push_back({mi, (int32_t)c});
  int rc = PSGD_OK;
  if (!rc) rc = rk_alloc(&rk->d_probs, rk->nprob, "rtopk problems");
  if (!rc) rc = rk_alloc(&rk->d_state, rk->nprob, "rtopk state");
  if (!rc) rc = rk_alloc(&rk->d_hist, (int64_t)rk->nprob * kRkBins, "rtopk histograms");
  if (!rc) rc = rk_alloc(&rk->d_arrive, rk->nprob, "rtopk counters");
  if (!rc) rc = rk_alloc(&rk->d_htiles, (int64_t)rk->htiles.size(), "rtopk tiles");
  if (!rc) rc = rk_alloc(&rk->d_ltiles, (int64_t)rk->ltiles.size(), "rtopk tiles");
  if (!rc) rc = rk_alloc(&rk->d_ccount, rk->nchunk_total, "rtopk chunk counts");
  if (!rc) rc = rk_alloc(&rk->d_sidx, rk->msg_total, "rtopk message indices");
  if (!rc) rc = rk_alloc(&rk->d_sval, rk->msg_total, "rtopk message values");
  if (rc) {
    rtopk_destroy(rk);
    return rc;
  }
  auto setup = [&]() -> int {
    if (!rk->hp.empty())
      CUDA_TRY(cudaMemcpy(rk->d_probs, rk->hp.data(), rk->hp.size() * sizeof(RkProb), cudaMemcpyHostToDevice));
    if (!rk->htiles.empty())
      CUDA_TRY(cudaMemcpy(rk->d_htiles, rk->htiles.data(), rk->htiles.size() * sizeof(RkTile), cudaMemcpyHostToDevice));
    if (!rk->ltiles.empty())
      CUDA_TRY(cudaMemcpy(rk->d_ltiles, rk->ltiles.data(), rk->ltiles.size() * sizeof(RkTile), cudaMemcpyHostToDevice));
    CUDA_TRY(cudaMemset(rk->d_hist, 0, (size_t)std::max(rk->nprob, 1) * kRkBins * sizeof(uint32_t)));
    CUDA_TRY(cudaMemset(rk->d_arrive, 0, (size_t)std::max(rk->nprob, 1) * sizeof(unsigned)));
    CUDA_TRY(cudaMemset(rk->d_sidx, 0, (size_t)std::max<int64_t>(rk->msg_total, 1) * sizeof(int32_t)));
    CUDA_TRY(cudaMemset(rk->d_sval, 0, (size_t)std::max<int64_t>(rk->msg_total, 1) * sizeof(float)));
    return PSGD_OK;
  };
  if ((rc = setup())) {
    rtopk_destroy(rk);
    return rc;
  }
  *out = rk;
  return PSGD_OK;
}

int rtopk_step(RTopK* rk, const float* const* G, float* B, int64_t total, float* U, int64_t step, cudaStream_t s) {
  RkArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int w = 0; w < rk->W; ++w) a.G[w] = G[w];
  a.B = B;
  a.U = U;
  a.total = total;
  a.layers = rk->d_layers;
  a.probs = rk->d_probs;
  a.state = rk->d_state;
  a.hist = rk->d_hist;
  a.arrive = rk->d_arrive;
  a.ccount = rk->d_ccount;
  a.sidx = rk->d_sidx;
  a.sval = rk->d_sval;
  a.W = rk->W;
  a.nmat = rk->nmat;
  a.seed = rk->seed;
  a.step = step;
  if (U) CUDA_TRY(cudaMemsetAsync(U, 0, (size_t)total * sizeof(float), s));
  if (rk->nprob > 0) {
    rk_begin_kernel<<<(rk->nprob + 127) / 128, 128, 0, s>>>(a, rk->nprob);
    CUDA_TRY(cudaGetLastError());
    a.tiles = rk->d_htiles;
    for (int draw = 0; draw < 2; ++draw)
      for (int q = 0; q < kRkPasses; ++q) {
        rk_hist_kernel<<<(unsigned)rk->htiles.size(), kRkThreads, 0, s>>>(a, q, draw);
        CUDA_TRY(cudaGetLastError());
      }
    a.tiles = rk->d_ltiles;
    rk_count_kernel<<<(unsigned)rk->ltiles.size(), kRkThreads, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
    rk_scan_kernel<<<(unsigned)rk->nprob, kRkThreads, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
    rk_apply_kernel<<<(unsigned)rk->ltiles.size(), kRkThreads, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
  }
  if (U && rk->nvec > 0) {
    rk_vec_kernel<<<64, 256, 0, s>>>(rk->d_vecs, rk->nvec, a);
    CUDA_TRY(cudaGetLastError());
  }
  return PSGD_OK;
}

int64_t rtopk_k(const RTopK* rk, int mi) { return rk->kk[mi]; }

void rtopk_message(const RTopK* rk, int mi, int w, const int32_t** idx, const float** val) {
  const RkProb& P = rk->hp[(size_t)w * rk->nmat + mi];
  *idx = rk->d_sidx + P.msg_off;
  *val = rk->d_sval + P.msg_off;
}

int rtopk_launches(const RTopK* rk) { return rk->nprob > 0 ? 1 + 2 * kRkPasses + 3 + (rk->nvec > 0 ? 1 : 0) : 1; }

}  // namespace psgd
