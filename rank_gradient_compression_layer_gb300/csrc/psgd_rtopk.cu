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
// digits per select; each round counts the digit of the entries still
// matching the prefix found so far and picks the bin that holds the key
// still needed (a select whose chosen bin holds exactly the entries still
// needed is finished early).
//
// Only pass 0 reads the whole layer: it forms M, counts the top digit of
// |M| (and the second one, near the previous step's top digit) and records
// the largest |M| of every 32 entries.  It is persistent: each CTA takes a
// contiguous run of tiles and arrives once per problem it touches, with the
// number of tiles it did.  Pass 1 reads only the groups of 32 whose largest
// |M| reaches the digits pass 0 chose, and lists the entries above them --
// members of T for sure -- and, with their values, those equal to them, the
// candidates.  A tail kernel (one CTA per problem, so its passes need no
// grid-wide hand-off) finishes the magnitude select over the candidates,
// completes the list of T with its draws, runs the draw select over it,
// sets the sent entries K in a bitmap (one bit per packed position) and
// turns their per-span counts into message offsets.  The apply kernel then
// writes the messages, E and U from the bitmaps and clears them for the
// next step.
#include <cuda_runtime.h>

#include <cstring>
#include <vector>

#include "psgd_kernels.cuh"
#include "psgd_plan.h"
#include "psgd_rtopk.h"

namespace psgd {
namespace {

constexpr int kRkThreads = 256;
constexpr int kRkGroups = 8;                           // float4 groups per thread (full passes)
constexpr int kRkChunk = kRkThreads * kRkGroups * 4;   // packed positions per full-pass tile
constexpr int kRkApplyWords = kRkThreads;              // bitmap words per apply tile (1 per thread)
constexpr int kRkSpan = kRkApplyWords * 32;            // packed positions per apply tile / count chunk
constexpr int kRkTail = 1024;                          // threads of the per-problem tail CTA
constexpr int kRkBins = 2048;                          // digits of at most 11 bits
constexpr int kRkPasses = 6;
// Digit layouts.  Magnitude keys: the first digit is bits 63..53 (bit 63 is
// |M|'s sign, clear), i.e. |M|'s exponent and top 2 mantissa bits; the
// second, bits 52..43, is the one pass 0 resolves too when it can (below).
// Draw keys: six digits over all 64 bits.
__constant__ int c_mshift[kRkPasses] = {53, 43, 32, 21, 10, 0};
__constant__ int c_mwidth[kRkPasses] = {11, 10, 11, 11, 11, 10};
__constant__ int c_dshift[kRkPasses] = {53, 42, 31, 20, 9, 0};
__constant__ int c_dwidth[kRkPasses] = {11, 11, 11, 11, 11, 9};
// Under error feedback many entries pile up just below the threshold, so
// the threshold's first-digit bin holds several percent of a layer, all
// candidates.  The bin moves little from step to step: pass 0 also counts
// the second digit of the entries whose first digit is within one of the
// previous step's (kRkWin bins of kRkFine sub-bins), and when this step's
// first digit lands there, both digits are known before pass 1.
constexpr int kRkWin = 3;
constexpr int kRkFine = 1024;           // second magnitude digit: 10 bits
constexpr int kRkTopBins = kRkBins + kRkWin * kRkFine;  // pass 0's counters per problem
constexpr uint32_t kRkNoTop = 0xFFFFFFFFu;
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

struct RkProb {   // one (worker, matrix layer) problem
  int32_t mi, w;  // matrix layer position, worker
  int64_t d, r, k;
  int64_t len;     // packed positions n x ld
  int64_t nchunks; // full-pass tiles (kRkChunk positions each)
  int64_t nwords;  // bitmap words, ceil(len / 32) (storage rounded up to 4; the rest stays 0)
  int64_t nspans;  // apply tiles / count chunks (kRkSpan positions each)
  int64_t chunk0;  // first span count of this problem
  int64_t msg_off; // first message entry of this problem
  int64_t list_off, bm_off;  // candidate list and list of T (capacity d each); K's bitmap
  int64_t host_off;          // its message in psgd_step_host's order (layer-major)
};

struct RkSel {      // one radix select
  uint64_t prefix;  // key bits found so far (the threshold once done)
  int64_t need;     // entries still to take from those matching the prefix
  int32_t done;     // the threshold is known
  int32_t pad;
};

struct RkState {
  RkSel sel[2];    // 0: the top set by magnitude (T = {Km >= threshold});
                   // 1: the draw among T (K = {Kr <= threshold})
  uint64_t dkey;   // draw stream key of this step
  unsigned long long counts;  // pass 1's list lengths: candidates (low 32 bits), sure members of T (high)
  uint32_t nT;     // members of T (the tail's list)
  uint32_t depth;  // magnitude digits pass 0 resolved (1 or 2)
  uint32_t prev_top;  // the first magnitude digit of the previous step (kRkNoTop: none); kept across steps
  uint32_t pad;
};

struct RkDraw {  // a member of T in the tail's list: flat index, draw h(i)
  uint32_t i, h;
};

struct RkCand {  // a candidate: flat index and M
  uint32_t i;
  float m;
};

struct RkTile {
  int32_t p;      // problem, or matrix layer (apply)
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
  uint32_t* hist;     // problems x kRkTopBins: pass 0's first-digit and windowed second-digit counts
  unsigned* arrive;   // problems
  const RkTile* tiles;
  int32_t ntiles;     // tiles of the kernel
  uint32_t* bm;       // bitmaps of K (zero between steps)
  uint32_t* wmax;     // per bitmap word: the largest |M| bit pattern among its entries (pass 0)
  RkCand* cand;       // candidate lists
  RkDraw* tlist;      // lists of T
  int64_t* ccount;    // per problem span counts of K, then their exclusive offsets
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

__device__ __forceinline__ uint64_t key_mag(float m, uint32_t i) {
  const uint32_t pat = __float_as_uint(m) & 0x7FFFFFFFu;
  return ((uint64_t)pat << 32) | (uint64_t)(0xFFFFFFFFu - i);
}

// h(i): the upper 32 bits of the draw stream at entry i (the draw key is (h(i), i)).
__device__ __forceinline__ uint32_t draw_hi(uint64_t dkey, uint32_t i) {
  return (uint32_t)(mix64(dkey + (uint64_t)(i + 1) * kGamma) >> 32);
}

__device__ __forceinline__ uint64_t mask_above(int shift, int width) {
  return shift + width >= 64 ? 0ull : (~0ull << (shift + width));
}

// Flat index of packed position p (relative to the layer; p < 2^31).
__device__ __forceinline__ uint32_t flat_of(const LayerDev& L, uint32_t p) {
  if (L.ld == L.m) return p;
  const uint32_t row = p / (uint32_t)L.ld;
  return p - row * (uint32_t)(L.ld - L.m);
}

// Packed position of flat index i.
__device__ __forceinline__ uint32_t packed_of(const LayerDev& L, uint32_t i) {
  if (L.ld == L.m) return i;
  const uint32_t row = i / (uint32_t)L.m;
  return i + row * (uint32_t)(L.ld - L.m);
}

// Exclusive prefix sum over the NT threads of the CTA (warp shuffles, then
// one warp over the warp totals: two barriers).  s_w: NT / 32 words of
// shared scratch; *all receives the total.  All threads call it.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_w, uint32_t* all) {
  constexpr int NW = NT / 32;
  static_assert(NW <= 32, "one warp scans the warp totals");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t x = lane < NW ? s_w[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane < NW) s_w[lane] = x;
  }
  __syncthreads();
  *all = s_w[NW - 1];
  const uint32_t r = incl - v + (warp ? s_w[warp - 1] : 0u);
  __syncthreads();  // s_w may be reused at once
  return r;
}

// Pick the digit at `shift` of the need-th key (largest first for the top
// set, smallest first for the draw) from the pass histogram h and narrow the
// select.  All NT threads of the CTA call it.  Counts fit 32 bits (a problem
// has fewer than 2^31 entries).
template <int NT>
__device__ void rk_find(RkSel& st, const uint32_t* h, int shift, int width, bool largest, uint32_t* s_w) {
  auto bin = [&](int b) -> uint32_t { return h[b]; };
  const int t = threadIdx.x;
  const int nb = 1 << width;
  const int per = (nb + NT - 1) / NT;
  // thread t owns walk positions [t per, t per + per); walk position j is
  // bin nb - 1 - j (largest first) or bin j (smallest first)
  uint32_t mine = 0;
  for (int j = t * per; j < t * per + per && j < nb; ++j) mine += bin(largest ? nb - 1 - j : j);
  // read before the scan's barriers: the thread that finds the digit
  // rewrites st right after them
  const uint64_t need = (uint64_t)st.need;
  uint32_t all;
  const uint32_t excl = block_excl_scan<NT>(mine, s_w, &all), incl = excl + mine;
  const uint64_t above = (shift + width >= 64) ? 0ull : (~0ull << (shift + width));
  const uint64_t below = (1ull << shift) - 1ull;  // bits under this digit
  if (need > all) {
    // every entry matching the prefix is taken: the threshold is the lowest
    // (largest first) or highest (smallest first) key with that prefix
    if (t == 0) {
      st.prefix = largest ? (st.prefix & above) : ((st.prefix & above) | ~above);
      st.done = 1;
    }
    return;
  }
  if (excl < need && need <= incl) {
    uint32_t c = excl;
    for (int j = t * per; j < t * per + per && j < nb; ++j) {
      const int b = largest ? nb - 1 - j : j;
      const uint32_t hb = bin(b);
      if (c + hb >= need) {
        const int64_t left = (int64_t)(need - c);
        st.prefix = (st.prefix & above) | ((uint64_t)b << shift);
        st.need = left;
        if ((uint64_t)left == hb) {  // the whole bin is taken: the bin's end is the threshold
          if (!largest) st.prefix |= below;
          st.done = 1;
        }
        break;
      }
      c += hb;
    }
  }
}

template <int NT, int NB = kRkBins>
__device__ __forceinline__ void rk_zero_hist(uint32_t* h) {
  for (int b = threadIdx.x; b < NB; b += NT) h[b] = 0u;
  __syncthreads();
}

// End of pass 0's run over problem p (`done` of its `total` tiles): merge
// the CTA's counts and, in the CTA that completes the problem, start its
// top-set select (need = r) with the first magnitude digit and, when it
// lies in the window counted at the second digit, that digit too; then
// reset the global counts and the list counters and keep the first digit
// for the next step's window.  h: kRkTopBins counters (first digit, then
// the window's second digit).
__device__ __noinline__ void rk_close_run(const RkArgs& a, int p, uint32_t win0, unsigned done, unsigned total,
                                          uint32_t* h, uint32_t* s_sum, int* s_flag) {
  __shared__ RkSel s_sel;
  uint32_t* gh = a.hist + (int64_t)p * kRkTopBins;
  __syncthreads();
  for (int b = threadIdx.x; b < kRkTopBins; b += kRkThreads)
    if (h[b]) atomicAdd(gh + b, h[b]);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atom_add_acq_rel(a.arrive + p, done);
    const bool last = (old + done == total);
    if (last) a.arrive[p] = 0u;
    *s_flag = last ? 1 : 0;
    if (last) s_sel = RkSel{0ull, a.probs[p].r, 0, 0};
  }
  __syncthreads();
  if (!*s_flag) return;
  static_assert((kRkChunk / 32) == 32 * (kRkThreads / 32), "pass 1: a warp per 32 words of a tile");
  static_assert(kRkTopBins % kRkThreads == 0, "whole rows of counters per thread");
  {
    uint32_t v[kRkTopBins / kRkThreads];  // all loads in flight at once
#pragma unroll
    for (int k = 0; k < kRkTopBins / kRkThreads; ++k) v[k] = __ldcg(gh + threadIdx.x + k * kRkThreads);
#pragma unroll
    for (int k = 0; k < kRkTopBins / kRkThreads; ++k) {
      h[threadIdx.x + k * kRkThreads] = v[k];
      gh[threadIdx.x + k * kRkThreads] = 0u;
    }
  }
  __syncthreads();
  rk_find<kRkThreads>(s_sel, h, c_mshift[0], c_mwidth[0], true, s_sum);
  __syncthreads();
  const uint32_t top = (uint32_t)(s_sel.prefix >> c_mshift[0]);
  const uint32_t slot = top - win0;  // the window's sub-histogram of this first digit, if counted
  uint32_t depth = 1;
  if (!s_sel.done && win0 != kRkNoTop && slot < (uint32_t)kRkWin) {
    rk_find<kRkThreads>(s_sel, h + kRkBins + slot * kRkFine, c_mshift[1], c_mwidth[1], true, s_sum);
    __syncthreads();
    depth = 2;
  }
  if (threadIdx.x == 0) {
    a.state[p].sel[0] = s_sel;
    a.state[p].counts = 0ull;
    a.state[p].depth = depth;
    a.state[p].prev_top = top;
  }
}

// Valid lanes of float4 group g of layer L (the padding of a row is not an entry).
__device__ __forceinline__ unsigned group_valid(const LayerDev& L, uint32_t g) {
  if (L.ld == L.m) return 0xFu;
  const uint32_t row = g / (uint32_t)L.F;
  const int col = 4 * (int)(g - row * (uint32_t)L.F);
  const int n = min(4, L.m - col);
  return (1u << n) - 1u;
}

__device__ __forceinline__ float comp(const float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// This CTA's contiguous run of pass 0's tiles.
__device__ __forceinline__ void rk_run(const RkArgs& a, int* t0, int* t1) {
  *t0 = (int)((int64_t)blockIdx.x * a.ntiles / gridDim.x);
  *t1 = (int)((int64_t)(blockIdx.x + 1) * a.ntiles / gridDim.x);
}

// Pass 0 (persistent, tiles in order): M = G + E into B, the top digit of
// |M| (and the second, near the previous step's top digit), the largest |M|
// of every bitmap word, and (worker 0's problems) U zeroed.
__global__ void __launch_bounds__(kRkThreads, 4) rk_pass0_kernel(RkArgs a) {
  __shared__ uint32_t h[kRkTopBins];  // first digit, then the window's second digit
  __shared__ uint32_t s_sum[kRkThreads / 32];
  __shared__ int s_flag;
  int t, t1;
  rk_run(a, &t, &t1);
  while (t < t1) {
    const RkTile first = a.tiles[t];
    const RkProb P = a.probs[first.p];
    const LayerDev L = a.layers[P.mi];
    const int te = (int)min((int64_t)t1, t + (P.nchunks - first.chunk));
    rk_zero_hist<kRkThreads, kRkTopBins>(h);
    // the window: first digits prev_top - 1 .. prev_top + 1 (none before the first step)
    const uint32_t prev = a.state[first.p].prev_top;
    const uint32_t win0 = prev == kRkNoTop ? kRkNoTop : prev - 1u;
    const uint32_t ng = (uint32_t)(P.len / 4);
    const float4* G4 = reinterpret_cast<const float4*>(a.G[P.w] + L.off);
    float4* B4 = reinterpret_cast<float4*>(a.B + (int64_t)P.w * a.total + L.off);
    float4* U4 = (a.U && P.w == 0) ? reinterpret_cast<float4*>(a.U + L.off) : nullptr;
    uint32_t* wmax = a.wmax + P.bm_off;
    constexpr int kHalf = kRkGroups / 2;
#pragma unroll 1
    for (int c = first.chunk; c < first.chunk + (te - t); ++c) {
      const uint32_t base = (uint32_t)c * (kRkThreads * kRkGroups) + threadIdx.x;
#pragma unroll 1
      for (int jb = 0; jb < kRkGroups; jb += kHalf) {
        float4 gv[kHalf], bv[kHalf];
#pragma unroll
        for (int u = 0; u < kHalf; ++u) {
          const uint32_t g = base + (uint32_t)(jb + u) * kRkThreads;
          if (g < ng) {
            gv[u] = __ldcs(G4 + g);
            bv[u] = B4[g];
          }
        }
#pragma unroll
        for (int u = 0; u < kHalf; ++u) {
          const uint32_t g = base + (uint32_t)(jb + u) * kRkThreads;
          uint32_t mx = 0;  // the group's largest |M| bit pattern
          if (g < ng) {
            const unsigned ok = group_valid(L, g);
            float4 mv = bv[u];
            if (ok & 1u) mv.x = gv[u].x + bv[u].x;
            if (ok & 2u) mv.y = gv[u].y + bv[u].y;
            if (ok & 4u) mv.z = gv[u].z + bv[u].z;
            if (ok & 8u) mv.w = gv[u].w + bv[u].w;
            B4[g] = mv;
            if (U4) U4[g] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (ok >> k & 1u) {
                const uint32_t pat = __float_as_uint(comp(mv, k)) & 0x7FFFFFFFu;
                mx = max(mx, pat);
                atomicAdd(&h[pat >> 21], 1u);
                const uint32_t slot = (pat >> 21) - win0;  // wraps (large) outside the window
                if (slot < (uint32_t)kRkWin) atomicAdd(&h[kRkBins + slot * kRkFine + ((pat >> 11) & (kRkFine - 1))], 1u);
              }
          }
          // the word's maximum over its 8 lanes (consecutive groups), for pass 1
          mx = max(mx, __shfl_xor_sync(kFull, mx, 1));
          mx = max(mx, __shfl_xor_sync(kFull, mx, 2));
          mx = max(mx, __shfl_xor_sync(kFull, mx, 4));
          if ((threadIdx.x & 7) == 0 && g < ng) wmax[g >> 3] = mx;
        }
      }
    }
    rk_close_run(a, first.p, win0, (unsigned)(te - t), (unsigned)P.nchunks, h, s_sum, &s_flag);
    t = te;
  }
}

// Pass 1: the list of the entries above the digits pass 0 resolved
// (members of T for sure) and the list of candidates (equal to them).  Only
// the bitmap words whose largest |M| reaches the candidates' range are
// read: with one percent of a layer in T, about a third of B.  One CTA per
// kRkP1Words words of a problem (last first: pass 0 wrote the end of B
// last, so it is still in L2); each warp owns 128 of them, finds the marked
// ones from the word maxima, and reads them 16 at a time (8 lanes per word,
// a float4 each), the next 16 in flight while it lists the current ones.
// The pass is latency bound: its CTAs are not persistent, so many keep
// loads in flight.
constexpr int kRkP1Words = 1024;
constexpr int kRkP1Sub = kRkP1Words / (kRkThreads / 32) / 32;  // 32-word blocks per warp (4)

__global__ void __launch_bounds__(kRkThreads) rk_pass1_kernel(RkArgs a) {
  __shared__ uint8_t s_words[kRkThreads / 32][32 * kRkP1Sub];  // each warp's marked words, in order
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RkTile tile = a.tiles[a.ntiles - 1 - blockIdx.x];
  const int p = tile.p;
  const RkProb P = a.probs[p];
  const LayerDev L = a.layers[P.mi];
  RkState* stp = a.state + p;
  const RkSel sel = stp->sel[0];
  const uint32_t ng = (uint32_t)(P.len / 4), nw = (uint32_t)P.nwords;
  const float4* B4 = reinterpret_cast<const float4*>(a.B + (int64_t)P.w * a.total + L.off);
  RkCand* cl = a.cand + P.list_off;
  RkDraw* sl = a.tlist + P.list_off;
  // |M| bit patterns: [lo, hi) holds the digits pass 0 resolved, >= hi is above
  // them (a finished select: everything from lo up is in T, no candidates)
  const uint32_t lo = (uint32_t)(sel.prefix >> 32);
  const uint32_t hi = sel.done ? lo : lo + (1u << (c_mshift[stp->depth - 1] - 32));
  const uint32_t w0 = (uint32_t)tile.chunk * kRkP1Words + (uint32_t)warp * (32 * kRkP1Sub);  // this warp's words
  int nall = 0;
  {
    uint32_t mx[kRkP1Sub];
#pragma unroll
    for (int b = 0; b < kRkP1Sub; ++b) {
      const uint32_t w = w0 + b * 32 + lane;
      mx[b] = w < nw ? __ldcg(a.wmax + P.bm_off + w) : 0u;
    }
    // the marked words listed in order: a marked lane writes its word at its rank
#pragma unroll
    for (int b = 0; b < kRkP1Sub; ++b) {
      const uint32_t w = w0 + b * 32 + lane;
      const bool mark = w < nw && mx[b] >= lo;
      const unsigned m = __ballot_sync(kFull, mark);
      if (mark) s_words[warp][nall + __popc(m & ((1u << lane) - 1u))] = (uint8_t)(b * 32 + lane);
      nall += __popc(m);
    }
    __syncwarp();
  }
  constexpr int kWords = 4;  // per lane group and batch: 4 groups of 8 lanes -> 16 words
  float4 cur[kWords], nxt[kWords];
  uint32_t gc[kWords], gn[kWords];
  auto fetch = [&](int batch, float4* v, uint32_t* gw) {
#pragma unroll
    for (int u = 0; u < kWords; ++u) {
      const int j = batch * 16 + (lane >> 3) + 4 * u;
      const int r = j < nall ? (int)s_words[warp][j] : -1;
      gw[u] = r >= 0 ? (w0 + (uint32_t)r) * 8 + (lane & 7) : 0xFFFFFFFFu;
      if (gw[u] < ng) v[u] = B4[gw[u]];
    }
  };
  const int nb = (nall + 15) / 16;
  if (nb > 0) fetch(0, cur, gc);
#pragma unroll 1
  for (int bt = 0; bt < nb; ++bt) {
    if (bt + 1 < nb) fetch(bt + 1, nxt, gn);
    unsigned smask = 0, cmask = 0;  // sure / candidate lanes, 4 bits per group
#pragma unroll
    for (int u = 0; u < kWords; ++u) {
      const unsigned ok = gc[u] < ng ? group_valid(L, gc[u]) : 0u;
      unsigned sure = 0, cnd = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t pat = __float_as_uint(comp(cur[u], k)) & 0x7FFFFFFFu;
        sure |= (pat >= hi ? 1u : 0u) << k;
        cnd |= (pat - lo < hi - lo ? 1u : 0u) << k;
      }
      smask |= (sure & ok) << (4 * u);
      cmask |= (cnd & ok) << (4 * u);
    }
    // one reservation per warp in both lists (a 64-bit counter pair)
    if (__any_sync(kFull, (smask | cmask) != 0)) {
      const uint32_t mine = ((uint32_t)__popc(smask) << 16) | (uint32_t)__popc(cmask);
      uint32_t incl = mine;  // <= 512 of each per warp: the halves never carry
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += x;
      }
      unsigned long long b0 = 0;
      if (lane == 31) b0 = atomicAdd(&stp->counts, ((unsigned long long)(incl >> 16) << 32) | (incl & 0xFFFFu));
      b0 = __shfl_sync(kFull, b0, 31);
      const uint32_t ex = incl - mine;
      uint32_t ss = (uint32_t)(b0 >> 32) + (ex >> 16);
      uint32_t cs = (uint32_t)b0 + (ex & 0xFFFFu);
#pragma unroll
      for (int u = 0; u < kWords; ++u) {
        const unsigned sm = (smask >> (4 * u)) & 0xFu, cm = (cmask >> (4 * u)) & 0xFu;
        if (!(sm | cm)) continue;
        const uint32_t g = gc[u];
        uint32_t i0;
        if (L.ld == L.m) {
          i0 = 4 * g;
        } else {
          const uint32_t row = g / (uint32_t)L.F;
          i0 = row * (uint32_t)L.m + 4 * (g - row * (uint32_t)L.F);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (sm >> k & 1u) sl[ss++] = RkDraw{i0 + k, 0u};
          if (cm >> k & 1u) cl[cs++] = RkCand{i0 + k, comp(cur[u], k)};
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kWords; ++u) {
      cur[u] = nxt[u];
      gc[u] = gn[u];
    }
  }
}

// The rest of one problem's selection, one CTA (kRkTail threads) per
// problem: magnitude digits 1.. over the candidates, the list of T
// completed (the sure members' draws, then the candidates that make T), the
// draw select over it, the sent entries set in K's bitmap and counted per
// span, and the spans' exclusive offsets.  Every loop keeps kRkBatch loads
// in flight per thread: one CTA has to cover a whole problem.
constexpr int kRkBatch = 8;

__global__ void __launch_bounds__(kRkTail, 1) rk_tail_kernel(RkArgs a) {
  __shared__ uint32_t h[kRkBins];
  __shared__ uint32_t s_sum[kRkTail / 32];
  __shared__ RkSel s_sel;
  __shared__ uint32_t s_cnt;
  const int p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const RkProb P = a.probs[p];
  const LayerDev L = a.layers[P.mi];
  RkState* stp = a.state + p;
  const unsigned long long cnts = stp->counts;
  const uint32_t nc = (uint32_t)cnts, ns = (uint32_t)(cnts >> 32);
  const RkCand* cl = a.cand + P.list_off;
  RkDraw* tl = a.tlist + P.list_off;
  uint32_t* bm = a.bm + P.bm_off;
  if (tid == 0) s_sel = stp->sel[0];
  __syncthreads();
  // the magnitude digits pass 0 left, over the candidates
  for (int q = (int)stp->depth; q < kRkPasses && !s_sel.done; ++q) {
    rk_zero_hist<kRkTail>(h);
    const int shift = c_mshift[q], width = c_mwidth[q];
    const uint64_t above = mask_above(shift, width), want = s_sel.prefix & above;
    const uint32_t dmask = (1u << width) - 1u;
    for (uint32_t e0 = tid; e0 < nc; e0 += kRkTail * kRkBatch) {
      RkCand cv[kRkBatch];
#pragma unroll
      for (int u = 0; u < kRkBatch; ++u)
        if (e0 + u * kRkTail < nc) cv[u] = cl[e0 + u * kRkTail];
#pragma unroll
      for (int u = 0; u < kRkBatch; ++u)
        if (e0 + u * kRkTail < nc) {
          const uint64_t K = key_mag(cv[u].m, cv[u].i);
          if ((K & above) == want) atomicAdd(&h[(uint32_t)(K >> shift) & dmask], 1u);
        }
    }
    __syncthreads();
    rk_find<kRkTail>(s_sel, h, shift, width, true, s_sum);
    __syncthreads();
  }
  const uint64_t vm = s_sel.prefix;
  const uint64_t step_key = mix64(a.seed + (uint64_t)(a.step + 1) * kGamma);
  const uint64_t dkey = mix64(step_key + (uint64_t)(P.w * 65536 + L.index + 1) * kGamma);
  __syncthreads();  // every thread has read vm
  if (tid == 0) {
    stp->sel[0] = s_sel;
    s_sel = RkSel{0ull, P.k, 0, 0};
    s_cnt = ns;
  }
  for (int b = tid; b < kRkBins; b += kRkTail) h[b] = 0u;
  __syncthreads();
  // the list of T with its draws, the top draw digit on the way: first the
  // sure members (in place) ...
  for (uint32_t e0 = tid; e0 < ns; e0 += kRkTail * kRkBatch) {
    uint32_t iv[kRkBatch];
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u)
      if (e0 + u * kRkTail < ns) iv[u] = tl[e0 + u * kRkTail].i;
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u)
      if (e0 + u * kRkTail < ns) {
        const uint32_t hv = draw_hi(dkey, iv[u]);
        tl[e0 + u * kRkTail].h = hv;
        atomicAdd(&h[hv >> 21], 1u);
      }
  }
  // ... then the candidates that make T, appended (warp-uniform batches, one
  // reservation per warp and batch)
  for (uint32_t eb = (uint32_t)(tid >> 5) * 32 * kRkBatch; eb < nc; eb += kRkTail * kRkBatch) {
    RkCand cv[kRkBatch];
    unsigned take = 0;
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u) {
      const uint32_t e = eb + u * 32 + lane;
      if (e < nc) cv[u] = cl[e];
    }
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u) {
      const uint32_t e = eb + u * 32 + lane;
      if (e < nc && key_mag(cv[u].m, cv[u].i) >= vm) take |= 1u << u;
    }
    const int n = __popc(take);
    int incl = n;
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += x;
    }
    uint32_t slot = 0;
    if (lane == 31 && incl) slot = atomicAdd(&s_cnt, (uint32_t)incl);
    slot = __shfl_sync(kFull, slot, 31) + (uint32_t)(incl - n);
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u)
      if (take >> u & 1u) {
        const uint32_t hv = draw_hi(dkey, cv[u].i);
        tl[slot++] = RkDraw{cv[u].i, hv};
        atomicAdd(&h[hv >> 21], 1u);
      }
  }
  __syncthreads();
  const uint32_t nT = s_cnt;
  rk_find<kRkTail>(s_sel, h, c_dshift[0], c_dwidth[0], false, s_sum);
  __syncthreads();
  for (int q = 1; q < kRkPasses && !s_sel.done; ++q) {
    rk_zero_hist<kRkTail>(h);
    const int shift = c_dshift[q], width = c_dwidth[q];
    const uint64_t above = mask_above(shift, width), want = s_sel.prefix & above;
    const uint32_t dmask = (1u << width) - 1u;
    for (uint32_t e0 = tid; e0 < nT; e0 += kRkTail * kRkBatch) {
      RkDraw dv[kRkBatch];
#pragma unroll
      for (int u = 0; u < kRkBatch; ++u)
        if (e0 + u * kRkTail < nT) dv[u] = tl[e0 + u * kRkTail];
#pragma unroll
      for (int u = 0; u < kRkBatch; ++u)
        if (e0 + u * kRkTail < nT) {
          const uint64_t K = ((uint64_t)dv[u].h << 32) | dv[u].i;
          if ((K & above) == want) atomicAdd(&h[(uint32_t)(K >> shift) & dmask], 1u);
        }
    }
    __syncthreads();
    rk_find<kRkTail>(s_sel, h, shift, width, false, s_sum);
    __syncthreads();
  }
  const uint64_t vr = s_sel.prefix;
  // K: the sent entries set in the bitmap (zero since the last apply) and
  // counted per span (in the free histogram when there are at most kRkBins
  // spans)
  int64_t* cc = a.ccount + P.chunk0;
  const bool local = P.nspans <= kRkBins;
  for (int c = tid; c < kRkBins; c += kRkTail) h[c] = 0u;
  if (!local)
    for (int64_t c = tid; c < P.nspans; c += kRkTail) cc[c] = 0;
  __syncthreads();
  for (uint32_t e0 = tid; e0 < nT; e0 += kRkTail * kRkBatch) {
    RkDraw dv[kRkBatch];
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u)
      if (e0 + u * kRkTail < nT) dv[u] = tl[e0 + u * kRkTail];
#pragma unroll
    for (int u = 0; u < kRkBatch; ++u)
      if (e0 + u * kRkTail < nT && (((uint64_t)dv[u].h << 32) | dv[u].i) <= vr) {
        const uint32_t pp = packed_of(L, dv[u].i);
        atomicOr(bm + (pp >> 5), 1u << (pp & 31));
        if (local)
          atomicAdd(&h[pp / kRkSpan], 1u);
        else
          atomicAdd(reinterpret_cast<unsigned long long*>(cc + pp / kRkSpan), 1ull);
      }
  }
  __syncthreads();
  // exclusive offsets of the span counts
  const int64_t per = (P.nspans + kRkTail - 1) / kRkTail;
  const int64_t b0 = tid * per, b1 = min(P.nspans, b0 + per);
  uint32_t mine = 0;
  for (int64_t b = b0; b < b1; ++b) mine += local ? h[b] : (uint32_t)__ldcg(cc + b);
  uint32_t tot;
  int64_t run = block_excl_scan<kRkTail>(mine, s_sum, &tot);
  for (int64_t b = b0; b < b1; ++b) {
    const int64_t x = local ? (int64_t)h[b] : __ldcg(cc + b);
    cc[b] = run;
    run += x;
  }
  if (tid == 0) {
    stp->sel[1] = s_sel;
    stp->dkey = dkey;
    stp->nT = nT;
  }
}

constexpr int kRkApplyFastW = 8;  // workers the apply kernel handles with all words in registers

// Messages, error and update of layer mi over one span, all workers in
// order: thread = one bitmap word (the scattered reads and writes of the
// sent entries are latency-bound, so one word per thread keeps the most of
// them in flight); the sent entries go to the worker's message at their
// index-ordered position, are zeroed in B (E = M - S) and summed into U
// (zeroed by pass 0), which is then scaled by 1 / W; the bitmap words are
// cleared.  The workers' records and span offsets are read once into shared
// memory.  Up to kRkApplyFastW workers, all their words are loaded at once
// and each sent entry is handled with every worker's load in flight; with
// more, the workers go one by one, the next one's word fetched while one is
// written.
__global__ void __launch_bounds__(kRkThreads) rk_apply_kernel(RkArgs a) {
  __shared__ int s_warp[kRkThreads / 32];
  __shared__ int64_t s_at[kMaxWorkers], s_end[kMaxWorkers], s_bm[kMaxWorkers];
  const RkTile t = a.tiles[blockIdx.x];
  const int mi = t.p;
  const LayerDev L = a.layers[mi];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < a.W) {
    const RkProb P = a.probs[threadIdx.x * a.nmat + mi];
    s_at[threadIdx.x] = P.msg_off + a.ccount[P.chunk0 + t.chunk];
    s_end[threadIdx.x] = P.msg_off + P.k;  // exactly k entries are selected; never write past them
    s_bm[threadIdx.x] = P.bm_off;
  }
  __syncthreads();
  const uint32_t w = (uint32_t)t.chunk * kRkApplyWords + threadIdx.x;
  const uint32_t nw = (uint32_t)(((int64_t)L.n * L.ld + 31) / 32);  // same for every worker
  const bool in = w < nw;
  float* Ul = a.U ? a.U + L.off : nullptr;
  if (a.W <= kRkApplyFastW) {
    // all workers' words at once, their ranks by block scans with no scattered
    // access in between (two workers per scan, 16 bits each: a CTA has at most
    // 8192 sent entries per worker), then every sent entry of the word with all
    // workers' loads in flight together; U is stored once, summed in worker order
    uint32_t K[kRkApplyFastW];
    int64_t at0[kRkApplyFastW];
#pragma unroll
    for (int wk = 0; wk < kRkApplyFastW; ++wk) K[wk] = (wk < a.W && in) ? __ldcg(a.bm + s_bm[wk] + w) : 0u;
#pragma unroll
    for (int wk = 0; wk < kRkApplyFastW; wk += 2) {
      if (wk >= a.W) break;
      uint32_t tot;
      const uint32_t ex = block_excl_scan<kRkThreads>((uint32_t)__popc(K[wk]) | ((uint32_t)__popc(K[wk + 1]) << 16),
                                                      reinterpret_cast<uint32_t*>(s_warp), &tot);
      at0[wk] = s_at[wk] + (ex & 0xFFFFu);
      at0[wk + 1] = wk + 1 < a.W ? s_at[wk + 1] + (ex >> 16) : 0;
    }
    uint32_t uni = 0;
#pragma unroll
    for (int wk = 0; wk < kRkApplyFastW; ++wk) uni |= K[wk];
    const float inv = 1.0f / (float)a.W;
    for (uint32_t bits = uni; bits; bits &= bits - 1) {
      const int b = __ffs(bits) - 1;
      const uint32_t pp = w * 32 + (uint32_t)b;
      const uint32_t below = (1u << b) - 1u;
      float v[kRkApplyFastW];
#pragma unroll
      for (int wk = 0; wk < kRkApplyFastW; ++wk)
        v[wk] = (K[wk] >> b & 1u) ? a.B[(int64_t)wk * a.total + L.off + pp] : 0.f;
      float u = 0.f;
#pragma unroll
      for (int wk = 0; wk < kRkApplyFastW; ++wk)
        if (K[wk] >> b & 1u) {
          const int64_t at = at0[wk] + __popc(K[wk] & below);
          if (at < s_end[wk]) {
            a.sidx[at] = (int32_t)flat_of(L, pp);
            a.sval[at] = v[wk];
          }
          a.B[(int64_t)wk * a.total + L.off + pp] = 0.f;
          u += v[wk];
        }
      if (Ul) Ul[pp] = u * inv;
    }
#pragma unroll
    for (int wk = 0; wk < kRkApplyFastW; ++wk)
      if (K[wk]) a.bm[s_bm[wk] + w] = 0u;  // K's bitmap is zero again for the next step
    return;
  }
  uint32_t uni = 0;
  uint32_t nxt = in ? __ldcg(a.bm + s_bm[0] + w) : 0u;
  for (int wk = 0; wk < a.W; ++wk) {
    const uint32_t K = nxt;
    if (wk + 1 < a.W && in) nxt = __ldcg(a.bm + s_bm[wk + 1] + w);
    const int c = __popc(K);
    // exclusive rank of this word's first sent entry within the span
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
    if (!c) continue;
    a.bm[s_bm[wk] + w] = 0u;  // K's bitmap is zero again for the next step
    int64_t at = s_at[wk] + base + incl - c;
    const int64_t end = s_end[wk];
    float* Bw = a.B + (int64_t)wk * a.total + L.off;
    for (uint32_t bits = K; bits; bits &= bits - 1) {
      const uint32_t pp = w * 32 + (uint32_t)(__ffs(bits) - 1);
      const float v = Bw[pp];
      if (at < end) {
        a.sidx[at] = (int32_t)flat_of(L, pp);
        a.sval[at] = v;
      }
      ++at;
      Bw[pp] = 0.f;
      if (Ul) Ul[pp] += v;
    }
    uni |= K;
  }
  if (Ul && uni) {
    const float inv = 1.0f / (float)a.W;
    for (uint32_t bits = uni; bits; bits &= bits - 1) {
      const uint32_t pp = w * 32 + (uint32_t)(__ffs(bits) - 1);
      Ul[pp] *= inv;
    }
  }
}

// Every problem's message into one buffer, layer-major: k indices (int32
// bits), then k values; grid.y = problem.
__global__ void rk_pack_kernel(const RkProb* probs, const int32_t* sidx, const float* sval, float* dst) {
  const RkProb P = probs[blockIdx.y];
  float* d = dst + P.host_off;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < P.k; e += (int64_t)gridDim.x * blockDim.x) {
    d[e] = __int_as_float(sidx[P.msg_off + e]);
    d[P.k + e] = sval[P.msg_off + e];
  }
}

// Vector layers: U = the worker mean; grid.y = vector layer.
__global__ void rk_vec_kernel(const VecDev* vecs, RkArgs a) {
  const VecDev V = vecs[blockIdx.y];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < V.n; i += (int64_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < a.W; ++w) s += a.G[w][V.off + i];
    a.U[V.off + i] = s / (float)a.W;
  }
}

}  // namespace

struct RTopK {
  int W = 0, nmat = 0, nprob = 0;
  uint64_t seed = 0;
  std::vector<RkProb> hp;
  std::vector<int64_t> kk;  // k per matrix layer
  std::vector<RkTile> ftiles, ptiles, ltiles;
  int pgrid = 0;  // CTAs of the persistent pass 0
  const LayerDev* d_layers = nullptr;
  const VecDev* d_vecs = nullptr;
  int nvec = 0;
  RkProb* d_probs = nullptr;
  RkState* d_state = nullptr;
  uint32_t* d_hist = nullptr;
  unsigned* d_arrive = nullptr;
  RkTile* d_ftiles = nullptr;  // (problem, chunk): pass 0
  RkTile* d_ptiles = nullptr;  // (problem, block of kRkP1Words words): pass 1
  RkTile* d_ltiles = nullptr;  // (matrix layer, span): apply
  uint32_t* d_bm = nullptr;
  uint32_t* d_wmax = nullptr;
  RkCand* d_cand = nullptr;
  RkDraw* d_tlist = nullptr;
  int64_t* d_ccount = nullptr;
  int32_t* d_sidx = nullptr;
  float* d_sval = nullptr;
  int64_t nchunk_total = 0, msg_total = 0, cand_total = 0, bm_total = 0;
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

template <class T>
int rk_upload(T* d, const std::vector<T>& h) {
  if (!h.empty()) CUDA_TRY(cudaMemcpy(d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice));
  return PSGD_OK;
}

}  // namespace

void rtopk_destroy(RTopK* rk) {
  if (!rk) return;
  void* ptrs[] = {rk->d_probs, rk->d_state, rk->d_hist,  rk->d_arrive, rk->d_ftiles, rk->d_ptiles, rk->d_ltiles,
                  rk->d_bm,    rk->d_wmax,  rk->d_cand,  rk->d_tlist,  rk->d_ccount, rk->d_sidx,   rk->d_sval};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  delete rk;
}

int rtopk_create(RTopK** out, const std::vector<LayerDev>& hl, const std::vector<VecDev>& hv,
                 const LayerDev* d_layers, const VecDev* d_vecs, int W, uint64_t seed, int top_div,
                 int sample_div) {
  *out = nullptr;
  if (top_div < 1 || sample_div < 1) return fail(PSGD_ERR_INVALID, "rTop-k divisors must be >= 1");
  for (const LayerDev& L : hl)
    if ((int64_t)L.n * L.ld >= ((int64_t)1 << 31))
      return fail(PSGD_ERR_INVALID, "rTop-k needs layers of fewer than 2^31 packed entries");
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
    rk->kk.push_back(ceil_div(ceil_div(d, top_div), sample_div));
  }
  for (int w = 0; w < W; ++w)
    for (int mi = 0; mi < rk->nmat; ++mi) {
      const int32_t p = w * rk->nmat + mi;
      RkProb P;
      P.mi = mi;
      P.w = w;
      P.d = (int64_t)hl[mi].n * hl[mi].m;
      P.r = ceil_div(P.d, top_div);
      P.k = rk->kk[mi];
      P.len = (int64_t)hl[mi].n * hl[mi].ld;
      P.nchunks = ceil_div(P.len, kRkChunk);
      P.nwords = ceil_div(P.len, 32);
      P.nspans = ceil_div(P.len, kRkSpan);
      P.chunk0 = rk->nchunk_total;
      rk->nchunk_total += P.nspans;
      P.msg_off = rk->msg_total;
      rk->msg_total += P.k;
      P.list_off = rk->cand_total;
      rk->cand_total += P.d;
      P.bm_off = rk->bm_total;
      rk->bm_total += (P.nwords + 3) & ~(int64_t)3;  // 16-byte aligned, whole uint4 per apply thread
      rk->hp.push_back(P);
      for (int64_t c = 0; c < P.nchunks; ++c) rk->ftiles.push_back({p, (int32_t)c});
      for (int64_t c = 0; c < ceil_div(P.nwords, kRkP1Words); ++c) rk->ptiles.push_back({p, (int32_t)c});
    }
  for (int mi = 0; mi < rk->nmat; ++mi)
    for (int64_t c = 0; c < rk->hp[mi].nspans; ++c) rk->ltiles.push_back({mi, (int32_t)c});
  {
    int64_t at = 0;  // psgd_step_host's message: layer-major, then worker
    for (int mi = 0; mi < rk->nmat; ++mi)
      for (int w = 0; w < W; ++w) {
        RkProb& P = rk->hp[(size_t)w * rk->nmat + mi];
        P.host_off = at;
        at += 2 * P.k;
      }
  }
  int rc = PSGD_OK;
  if (!rc) rc = rk_alloc(&rk->d_probs, rk->nprob, "rtopk problems");
  if (!rc) rc = rk_alloc(&rk->d_state, rk->nprob, "rtopk state");
  if (!rc) rc = rk_alloc(&rk->d_hist, (int64_t)rk->nprob * kRkTopBins, "rtopk histograms");
  if (!rc) rc = rk_alloc(&rk->d_arrive, rk->nprob, "rtopk counters");
  if (!rc) rc = rk_alloc(&rk->d_ftiles, (int64_t)rk->ftiles.size(), "rtopk tiles");
  if (!rc) rc = rk_alloc(&rk->d_ltiles, (int64_t)rk->ltiles.size(), "rtopk tiles");
  if (!rc) rc = rk_alloc(&rk->d_ptiles, (int64_t)rk->ptiles.size(), "rtopk tiles");
  if (!rc) rc = rk_alloc(&rk->d_bm, rk->bm_total, "rtopk bitmaps");
  if (!rc) rc = rk_alloc(&rk->d_wmax, rk->bm_total, "rtopk word maxima");
  if (!rc) rc = rk_alloc(&rk->d_cand, rk->cand_total, "rtopk candidate lists");
  if (!rc) rc = rk_alloc(&rk->d_tlist, rk->cand_total, "rtopk top-set lists");
  if (!rc) rc = rk_alloc(&rk->d_ccount, rk->nchunk_total, "rtopk chunk counts");
  if (!rc) rc = rk_alloc(&rk->d_sidx, rk->msg_total, "rtopk message indices");
  if (!rc) rc = rk_alloc(&rk->d_sval, rk->msg_total, "rtopk message values");
  if (rc) {
    rtopk_destroy(rk);
    return rc;
  }
  auto setup = [&]() -> int {
    int e = rk_upload(rk->d_probs, rk->hp);
    if (!e) e = rk_upload(rk->d_ftiles, rk->ftiles);
    if (!e) e = rk_upload(rk->d_ltiles, rk->ltiles);
    if (!e) e = rk_upload(rk->d_ptiles, rk->ptiles);
    if (e) return e;
    CUDA_TRY(cudaMemset(rk->d_bm, 0, (size_t)std::max<int64_t>(rk->bm_total, 1) * sizeof(uint32_t)));
    CUDA_TRY(cudaMemset(rk->d_hist, 0, (size_t)std::max(rk->nprob, 1) * kRkTopBins * sizeof(uint32_t)));
    CUDA_TRY(cudaMemset(rk->d_state, 0xFF, (size_t)std::max(rk->nprob, 1) * sizeof(RkState)));  // prev_top: none
    CUDA_TRY(cudaMemset(rk->d_arrive, 0, (size_t)std::max(rk->nprob, 1) * sizeof(unsigned)));
    CUDA_TRY(cudaMemset(rk->d_sidx, 0, (size_t)std::max<int64_t>(rk->msg_total, 1) * sizeof(int32_t)));
    CUDA_TRY(cudaMemset(rk->d_sval, 0, (size_t)std::max<int64_t>(rk->msg_total, 1) * sizeof(float)));
    // pass 0 is persistent: one wave of resident CTAs
    int dev = 0, sms = 0, o0 = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o0, rk_pass0_kernel, kRkThreads, 0));
    rk->pgrid = (int)std::min<int64_t>((int64_t)rk->ftiles.size(), (int64_t)sms * std::max(1, o0));
    return PSGD_OK;
  };
  if ((rc = setup())) {
    rtopk_destroy(rk);
    return rc;
  }
  *out = rk;
  return PSGD_OK;
}

int rtopk_step(RTopK* rk, const float* const* G, float* B, int64_t total, float* U, int64_t step, cudaStream_t s,
               const cudaEvent_t* ev) {
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
  a.bm = rk->d_bm;
  a.wmax = rk->d_wmax;
  a.cand = rk->d_cand;
  a.tlist = rk->d_tlist;
  a.ccount = rk->d_ccount;
  a.sidx = rk->d_sidx;
  a.sval = rk->d_sval;
  a.W = rk->W;
  a.nmat = rk->nmat;
  a.seed = rk->seed;
  a.step = step;
  auto mark = [&](int k) -> int {
    if (ev) CUDA_TRY(cudaEventRecord(ev[k], s));
    return PSGD_OK;
  };
  int rc;
  if (rk->nprob > 0) {
    a.tiles = rk->d_ftiles;
    a.ntiles = (int32_t)rk->ftiles.size();
    rk_pass0_kernel<<<(unsigned)rk->pgrid, kRkThreads, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
    if ((rc = mark(0))) return rc;
    a.tiles = rk->d_ptiles;
    a.ntiles = (int32_t)rk->ptiles.size();
    rk_pass1_kernel<<<(unsigned)rk->ptiles.size(), kRkThreads, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
    if ((rc = mark(1))) return rc;
    rk_tail_kernel<<<(unsigned)rk->nprob, kRkTail, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
    if ((rc = mark(2))) return rc;
    a.tiles = rk->d_ltiles;
    a.ntiles = (int32_t)rk->ltiles.size();
    rk_apply_kernel<<<(unsigned)rk->ltiles.size(), kRkThreads, 0, s>>>(a);
    CUDA_TRY(cudaGetLastError());
  } else {
    for (int k = 0; k < 3; ++k)
      if ((rc = mark(k))) return rc;
  }
  if (U && rk->nvec > 0) {
    rk_vec_kernel<<<dim3(16, (unsigned)rk->nvec), 256, 0, s>>>(rk->d_vecs, a);
    CUDA_TRY(cudaGetLastError());
  }
  return mark(3);
}

int64_t rtopk_k(const RTopK* rk, int mi) { return rk->kk[mi]; }

void rtopk_message(const RTopK* rk, int mi, int w, const int32_t** idx, const float** val) {
  const RkProb& P = rk->hp[(size_t)w * rk->nmat + mi];
  *idx = rk->d_sidx + P.msg_off;
  *val = rk->d_sval + P.msg_off;
}

int rtopk_pack(const RTopK* rk, float* dst, cudaStream_t s) {
  if (rk->nprob == 0) return PSGD_OK;
  rk_pack_kernel<<<dim3(8, (unsigned)rk->nprob), 256, 0, s>>>(rk->d_probs, rk->d_sidx, rk->d_sval, dst);
  CUDA_TRY(cudaGetLastError());
  return PSGD_OK;
}

int rtopk_launches(const RTopK* rk) {
  // passes 0 and 1, tail, apply (+ vectors)
  return (rk->nprob > 0 ? 4 : 0) + (rk->nvec > 0 ? 1 : 0);
}

}  // namespace psgd
