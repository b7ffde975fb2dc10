// Device code of the PowerSGD compression step for sm_103a.
//
// A step is four stream-ordered phase kernels (a fifth at r >= 8), each a
// plain grid of independent tiles over ALL layers of the context (one launch
// per phase, not per layer):
//
//   project         M_w = G_w + (B_w - Phat' Q_w'^T): B holds M of the last
//                   step, so the bracket is the error E_w; store B_w <- M_w;
//                   P rows = (sum_w M_w) Q.  The CTA that completes a row
//                   block writes its P rows and their Gram partial P^T P
//                   (float64); the CTA that completes a layer sums the Gram
//                   (fixed order), factors A = R^T R (Cholesky, float64),
//                   stores R and decides whether one Cholesky-QR pass is
//                   orthogonal enough (kappa_F(R) <= 1e3).  r >= 16: the
//                   tensor-core tile of psgd_mma.cuh; options.one_pass
//                   (r <= 4): the cluster kernel of psgd_cluster.cuh.
//   orthonormalise  rows P1 = P R^-1 by forward substitution (float64,
//                   rounded to float32, stored over P).  Where one pass is
//                   not enough (Cholesky-QR2), the CTA that completes the
//                   layer factors the Gram matrix of P1 the same way and
//                   stores X = R2^-1, so Phat = P1 X; at r >= 8 a fifth kernel
//                   stores those Phat rows once.
//   back-project    partial Q_w = M_w^T Phat over a row tile of one segment
//                   and one worker (at r <= 4 with the Phat rows formed from
//                   P1 and X as they are staged; one tile per row tile stores
//                   them); the CTA that completes (segment, worker) sums the
//                   partials (fixed order) into Q_w, and the one that
//                   completes the segment forms Qbar = mean_w Q_w.
//   decompress      U rows = Phat Qbar^T; vector layers U = mean_w G_w.
//
// The error buffer is never written as such: E_w = B_w - Phat Q_w^T is rebuilt
// on the fly by the next step's project phase (r FMAs per element), which
// saves a full read+write pass over every error buffer.
//
// The hot phases stream with 128-bit loads at high occupancy: an SM's share
// of GB300's HBM bandwidth (about 45 GB/s) over a loaded latency of one to two
// microseconds needs 50-100 KB in flight per SM, which many resident warps
// with a few independent loads each provide.  Every reduction runs in a fixed
// order, so a step is bit-reproducible.  Data written by another CTA of the
// same kernel is read with ld.global.cg (L2).
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "psgd_internal.h"

namespace psgd {

template <int RP>
struct Cfg {
  static constexpr int NG = RP * (RP + 1) / 2;              // Gram entries (upper triangle)
  // project: tiles of R1 rows x one segment x all workers; a warp per worker,
  // RSB rows per pass
  static constexpr int RSB = RP <= 4 ? 4 : (RP == 8 ? 2 : 1);
  static constexpr int R1 = 32;
  static constexpr int R1MAX = RP >= 16 ? 128 : R1;        // rows of a project row block at most (tensor-core tiles: 128)
  static constexpr int P1_WARPS = 8;                        // at most (more workers loop)
  static constexpr int P1_MINB = RP <= 2 ? 4 : (RP == 4 ? 3 : 1);          // 256-thread CTAs per SM the registers must allow
  // back-project: 8 warps over interleaved groups of UNR3 rows a warp loads
  // at once, and the CTAs per SM the registers must allow (more CTAs hide
  // each other's start-up and closing sums; two at r >= 16, whose
  // accumulators take the most registers)
  static constexpr int UNR3 = 8;
  static constexpr int P3_MINB = RP <= 2 ? 4 : (RP <= 8 ? 3 : 2);
  // decompress: RU rows x one segment per CTA of 256 threads
  static constexpr int RU = 128;
};

constexpr int kP1TRow = kSeg * 4 + 4;  // tiled project: shared row stride of the staged Q rows (floats)
constexpr int kP3Threads = 256;
constexpr int kUThreads = 256;

constexpr int kVChunk = 8192;  // vector elements per decompress tile
constexpr int kGramThreads = 128;  // split step: threads of a Gram tile
constexpr unsigned kFull = 0xffffffffu;

// ----------------------------------------------------------------------------
// helpers
// ----------------------------------------------------------------------------

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// A phase kernel's tile and layer record, staged in shared memory by the
// first warp before the programmatic-dependent wait, so that their two
// dependent round trips overlap the end of the phase before.  The tables are
// written before the step's first phase (by the host, or by a kernel the
// project phase waited for), so only a later phase may read them early, and
// it reads them through L2 (ld.global.cg): one request per table row and
// CTA, as lane i loads word i of the record (every thread loading the whole
// record would send the grid's requests for one layer to one L2 slice).
// The caller's barrier after the wait publishes them to the CTA.
struct EarlyTables {
  Tile t;
  LayerDev L;
};

__device__ __forceinline__ void stage_tables_early(const StepArgs& a, EarlyTables* s, bool vector_tiles) {
  static_assert(sizeof(Tile) == 16 && sizeof(LayerDev) % 8 == 0 && sizeof(LayerDev) / 8 <= 32,
                "a tile is one 16-byte word and a layer record at most 32 8-byte words");
  if (threadIdx.x >= 32) return;
  const int4 v = __ldcg(reinterpret_cast<const int4*>(a.tiles + blockIdx.x));
  const Tile t{v.x, v.y, v.z, v.w};
  if (threadIdx.x == 0) s->t = t;
  if (vector_tiles && t.c == 1) return;  // a vector tile: no layer record
  const int lane = (int)threadIdx.x;
  if (lane < (int)(sizeof(LayerDev) / 8))
    reinterpret_cast<long long*>(&s->L)[lane] = __ldcg(reinterpret_cast<const long long*>(a.layers + t.layer) + lane);
}

// An L2 cache policy under which the lines written are evicted last.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte store with an L2 cache policy.
__device__ __forceinline__ void st_policy_f4(float* addr, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Sums each of N values (N a power of two, 1..32) over the 32 lanes of a
// warp with N - 1 + 5 - log2(N) shuffles: every level of the butterfly hands
// half of the still-unsummed values to the partner lane, until each lane
// holds one value, then the remaining levels sum that value.  Afterwards the
// total of value j is held by lane j << (5 - log2 N) (and its group).
// Returns the lane's value index.  Deterministic: each total is formed by one
// fixed expression tree.
template <int N>
__device__ __forceinline__ int warp_reduce_multi(float (&v)[N], float& out) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
  const int lane = threadIdx.x & 31;
  constexpr int LOGN = N == 1 ? 0 : (N == 2 ? 1 : (N == 4 ? 2 : (N == 8 ? 3 : (N == 16 ? 4 : 5))));
  int idx = 0;
#pragma unroll
  for (int l = 0; l < LOGN; ++l) {
    const int o = 16 >> l;
    const int c = N >> l;  // values still held
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = up ? v[i] : v[i + c / 2];
      const float keep = up ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
    idx = (idx << 1) | (up ? 1 : 0);
  }
  float x = v[0];
#pragma unroll
  for (int o = 16 >> LOGN; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  out = x;
  return idx;
}

// (i, j), i <= j, of upper-triangle entry e in row-major order.
__device__ __forceinline__ void tri_index(int e, int rp, int& i, int& j) {
  i = 0;
  int rowlen = rp;
  while (e >= rowlen) {
    e -= rowlen;
    ++i;
    --rowlen;
  }
  j = i + e;
}

// Programmatic dependent launch (the phase kernels are launched as dependents
// of the kernel before them in the stream): wait until that kernel has
// completed and its writes are visible -- a no-op for a normal launch -- then
// let the next kernel's CTAs be scheduled while this grid runs, so they are
// resident and waiting when it ends.  Every phase kernel calls this before it
// reads anything a kernel of the step writes (the later phases stage their
// tile and layer record first: stage_tables_early).
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Whole CTA: make the CTA's global writes visible, count one arrival on *cnt
// and return true (in every thread) when this was arrival number `total`.
// The last arriver resets the counter for the next launch and may then read
// everything the other arrivers wrote (with .cg loads).  The barrier orders
// every thread's writes before thread 0's fence, whose cumulativity makes
// them visible at GPU scope before the arrival; one fence per CTA, not one
// per thread.
__device__ __forceinline__ bool cta_arrive_last(unsigned* cnt, unsigned total, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atom_add_acq_rel(cnt, 1u);
    const bool last = (old == total - 1);
    if (last) *cnt = 0u;
    *s_flag = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *s_flag != 0;
  __syncthreads();
  return last;
}

// Fused step: publish that what this CTA (or warp) wrote before is complete
// by raising *f to the step's epoch.  The caller has ordered the writes
// before this thread (barrier or __syncwarp); the fence makes them visible
// at GPU scope before the release store.
__device__ __forceinline__ void flag_raise(unsigned* f, unsigned epoch) {
  __threadfence();
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(epoch) : "memory");
}

// ----------------------------------------------------------------------------
// Gram-Schmidt coefficients from the Gram matrix (float64, warp-parallel)
// ----------------------------------------------------------------------------
//
// A = P^T P = R^T R with R upper triangular, diag > 0: R is the R factor of
// Gram-Schmidt on the columns of P, and Phat = P R^-1.  Lane j holds column j
// of A; step k takes the pivot from lane k, scales row k and updates the
// trailing columns (right-looking).  A pivot that is not positive marks a
// column whose remainder vanished: its row of R is zero and 1/R_kk is set to
// 0, so the matching column of Phat is zero.  Writes R (RP x RP, row-major)
// and 1/diag(R) to `out`.  One warp.
template <int RP>
__device__ void warp_cholesky(const double* A, double* out) {
  const int lane = threadIdx.x & 31;
  double a[RP];
#pragma unroll
  for (int i = 0; i < RP; ++i) a[i] = (lane < RP) ? A[i * RP + lane] : 0.0;
  double dinv = 0.0;
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    const double d = __shfl_sync(kFull, a[k], k);
    const bool deg = !(d > 0.0);
    const double rkk = deg ? 0.0 : sqrt(d);
    double rkj;
    if (lane == k)
      rkj = rkk;
    else if (lane > k && !deg)
      rkj = a[k] / rkk;
    else
      rkj = 0.0;
    if (lane == k) dinv = deg ? 0.0 : 1.0 / rkk;
    if (lane >= k) a[k] = rkj;
#pragma unroll
    for (int i = k + 1; i < RP; ++i) {
      const double rki = __shfl_sync(kFull, rkj, i);
      if (lane > k) a[i] -= rki * rkj;
    }
  }
  if (lane < RP) {
#pragma unroll
    for (int i = 0; i < RP; ++i) out[i * RP + lane] = (i <= lane) ? a[i] : 0.0;
    out[RP * RP + lane] = dinv;
  }
}

// Upper-triangular inverse X = R^-1 of the factor warp_cholesky left in
// fr (R row-major, then 1 / diag R), written to X (row-major).  Lane k < RP
// forms row k: X_kk = 1 / R_kk, X_kj = -(sum_{k <= l < j} X_kl R_lj) / R_jj.
// A column whose pivot was marked degenerate (1 / R_jj = 0) comes out zero.
template <int RP>
__device__ void warp_tri_inverse(const double* fr, double* X) {
  const int k = threadIdx.x & 31;
  if (k >= RP) return;
  double x[RP];
#pragma unroll
  for (int j = 0; j < RP; ++j) x[j] = 0.0;
#pragma unroll
  for (int j = 0; j < RP; ++j) {
    if (j == k) {
      x[j] = fr[RP * RP + j];
    } else if (j > k) {
      double s = 0.0;
#pragma unroll
      for (int l = 0; l < j; ++l)
        if (l >= k) s = fma(x[l], fr[l * RP + j], s);
      x[j] = -s * fr[RP * RP + j];
    }
  }
#pragma unroll
  for (int j = 0; j < RP; ++j) X[k * RP + j] = x[j];
}

// The CTA has stored the Gram partial of slot `slot` (of nslots) at
// gp + slot * NG.  The slots are summed in groups of kGramGroup (the group's
// last arriver, counter cgrp[group]; the group sum goes to slot nslots +
// group), then over the groups (the layer's last arriver); each sum in a
// fixed order.  The layer's last arriver factors the total: R (Cholesky),
// R^-1, and the flags of the factor record.  pub (fused step only): the
// layer's R flag, raised once R is stored.
template <int RP>
__device__ void gram_finish(const StepArgs& a, const LayerDev& L, double* gp, int slot, int nslots, unsigned* cgrp,
                            double* s_gram, int* s_flag, unsigned* pub) {
  constexpr int NG = Cfg<RP>::NG;
  const int grp = slot / kGramGroup;
  const int ngrp = (nslots + kGramGroup - 1) / kGramGroup;
  const int gsz = min(kGramGroup, nslots - grp * kGramGroup);
  if (!cta_arrive_last(cgrp + grp, (unsigned)gsz, s_flag)) return;
  for (int e = threadIdx.x; e < NG; e += blockDim.x) {
    double s = 0.0;
    for (int t = 0; t < gsz; ++t) s += __ldcg(gp + (int64_t)(grp * kGramGroup + t) * NG + e);
    gp[(int64_t)(nslots + grp) * NG + e] = s;
  }
  if (!cta_arrive_last(a.counters + L.cnt_off + L.c_gram, (unsigned)ngrp, s_flag)) return;
  for (int e = threadIdx.x; e < NG; e += blockDim.x) {
    double s = 0.0;
    for (int g = 0; g < ngrp; ++g) s += __ldcg(gp + (int64_t)(nslots + g) * NG + e);
    int i, j;
    tri_index(e, RP, i, j);
    s_gram[i * RP + j] = s;
    s_gram[j * RP + i] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    double* fr = a.rinv + L.rinv_off;
    warp_cholesky<RP>(s_gram, fr);
    __syncwarp();
    // Is one Cholesky-QR pass orthogonal enough?  Its loss of orthogonality
    // is about kappa(P)^2 eps; kappa_F = ||R||_F ||R^-1||_F bounds kappa(P).
    // At kappa_F <= 1e3 it is below 1e-9, far under Phat's float32 rounding,
    // and the second pass is skipped (flag X = I, Phat = P1).
    warp_tri_inverse<RP>(fr, s_gram);  // R^-1 (s_gram is free once the factor is taken)
    __syncwarp();
    double r2 = 0.0, x2 = 0.0;
    for (int e = threadIdx.x; e < RP * RP; e += 32) {
      r2 = fma(fr[e], fr[e], r2);
      x2 = fma(s_gram[e], s_gram[e], x2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      r2 += __shfl_xor_sync(kFull, r2, o);
      x2 += __shfl_xor_sync(kFull, x2, o);
    }
    // The one-pass back-project (Q_w = Y_w R^-1) when the project phase
    // formed Y and P is well conditioned: R^-1 goes to the X slot.
    const bool yk = a.ypath != 0 && r2 * x2 <= kYKappa2;
    if (yk)
      for (int e = threadIdx.x; e < RP * RP; e += 32) fr[RP * RP + RP + e] = s_gram[e];
    if (threadIdx.x == 0) {
      fr[2 * RP * RP + RP] = (r2 * x2 <= 1e6) ? 1.0 : 0.0;
      fr[2 * RP * RP + RP + 1] = yk ? 1.0 : 0.0;
    }
    if (pub) {
      __syncwarp();
      if (threadIdx.x == 0 && L.index != a.stall_layer) flag_raise(pub, a.epoch);
    }
  }
}

// CTA that completed row block rb of layer L (P rows in s_prow): Gram partial
// of the rows, then gram_finish over the layer's row blocks.
template <int RP>
__device__ void gram_tail(const StepArgs& a, const LayerDev& L, int rb, const float* s_prow, int nrows,
                          double* s_gram, int* s_flag, unsigned* pub) {
  constexpr int NG = Cfg<RP>::NG;
  double* gp = a.gram + L.gram_off;
  for (int e = threadIdx.x; e < NG; e += blockDim.x) {
    int i, j;
    tri_index(e, RP, i, j);
    double s = 0.0;
    for (int rr = 0; rr < nrows; ++rr) s = fma((double)s_prow[rr * RP + i], (double)s_prow[rr * RP + j], s);
    gp[(int64_t)rb * NG + e] = s;
  }
  gram_finish<RP>(a, L, gp, rb, L.nrb, a.counters + L.cnt_off + L.c_grp, s_gram, s_flag, pub);
}

// ----------------------------------------------------------------------------
// project: error add, B <- M, P = (sum_w M_w) Q, Gram
// ----------------------------------------------------------------------------
//
// A CTA owns R1 rows x one segment (128 columns) of one layer and all W
// workers; warp v handles workers v, v + 8, ...  Each lane holds its 4
// columns' rows of Q and of its worker's Q_w' in registers.

// Per-tile geometry and flags of the project phase.
struct P1Tile {
  int rb, seg, row0, rcnt, lane, warp, nwarps, c;
  bool act, tailc, prev, ub;  // ub: unbiased variant (M = G, B untouched)
};

template <int RP>
__device__ __forceinline__ P1Tile p1_tile(const StepArgs& a, const Tile& t, const LayerDev& L) {
  P1Tile T;
  T.rb = t.a;
  T.seg = t.b;
  T.row0 = T.rb * L.r1;
  T.rcnt = min(L.r1, L.n - T.row0);
  T.lane = threadIdx.x & 31;
  T.warp = threadIdx.x >> 5;
  T.nwarps = blockDim.x >> 5;
  T.c = T.seg * kSeg + T.lane;  // this lane's float4 column
  T.act = T.c < L.F;
  T.tailc = T.act && (T.c == L.F - 1) && (L.tail < 4);
  T.ub = a.unbiased != 0;
  T.prev = a.has_prev != 0 && !T.ub;
  return T;
}

// The RP values of rows 4c .. 4c + 3 of an ld x RP factor (Q or Q_w'),
// which sit contiguously: RP float4 loads per lane, coalesced over the warp.
template <int RP>
__device__ __forceinline__ void p1_load_q(const float* Qrows, const P1Tile& T, bool zero, float (&q)[4][RP]) {
  float* flat = &q[0][0];
  if (zero || !T.act) {
#pragma unroll
    for (int i = 0; i < 4 * RP; ++i) flat[i] = 0.f;
    return;
  }
  const float4* src = reinterpret_cast<const float4*>(Qrows + (int64_t)(4 * T.c) * RP);
#pragma unroll
  for (int i = 0; i < RP; ++i) {
    const float4 v = __ldg(src + i);
    flat[4 * i] = v.x;
    flat[4 * i + 1] = v.y;
    flat[4 * i + 2] = v.z;
    flat[4 * i + 3] = v.w;
  }
}

// The arithmetic of one pass over rn <= RSB rows of one worker, starting at
// tile row sb: the error E = B - Phat' Q_w'^T (k ascending, the same chain
// as the error read-back kernel; the previous Phat rows are warp-uniform
// loads), M = G + E stored to B, and the lane's share of the rows' P
// partials in acc.
template <int RP>
__device__ __forceinline__ void p1_rows(const LayerDev& L, const P1Tile& T, const float4 (&g)[Cfg<RP>::RSB],
                                        const float4 (&b)[Cfg<RP>::RSB], int sb, int rn, const float* Pprev,
                                        const float (&qv)[4][RP], const float (&qw)[4][RP], float* Bw,
                                        float (&acc)[Cfg<RP>::RSB * RP]) {
  constexpr int RSB = Cfg<RP>::RSB;
#pragma unroll
  for (int i = 0; i < RSB * RP; ++i) acc[i] = 0.f;
#pragma unroll
  for (int i = 0; i < RSB; ++i) {
    if (T.act && i < rn) {
      float e0 = b[i].x, e1 = b[i].y, e2 = b[i].z, e3 = b[i].w;
      if (T.prev) {
#pragma unroll
        for (int k = 0; k < RP; ++k) {
          const float p = __ldg(Pprev + (sb + i) * RP + k);
          e0 = fmaf(-p, qw[0][k], e0);
          e1 = fmaf(-p, qw[1][k], e1);
          e2 = fmaf(-p, qw[2][k], e2);
          e3 = fmaf(-p, qw[3][k], e3);
        }
      }
      float m0 = g[i].x + e0, m1 = g[i].y + e1, m2 = g[i].z + e2, m3 = g[i].w + e3;
      if (T.tailc) {
        if (L.tail < 2) m1 = 0.f;
        if (L.tail < 3) m2 = 0.f;
        m3 = 0.f;
      }
      if (!T.ub) {
        // rows the back-project reads first stay in L2 (evict-last); the
        // rest stream out (evict-first), leaving L2 to the loads in flight
        const int row = T.row0 + sb + i;
        float* dst = Bw + (int64_t)row * L.ld;
        if (row >= L.l2row)
          st_policy_f4(dst, make_float4(m0, m1, m2, m3), l2_evict_last_policy());
        else
          __stcs(reinterpret_cast<float4*>(dst), make_float4(m0, m1, m2, m3));
      }
#pragma unroll
      for (int k = 0; k < RP; ++k) {
        float t = m0 * qv[0][k];
        t = fmaf(m1, qv[1][k], t);
        t = fmaf(m2, qv[2][k], t);
        t = fmaf(m3, qv[3][k], t);
        acc[i * RP + k] = t;
      }
    }
  }
}

// The pass's P partials summed over the lanes into s_red_w (first worker of
// the warp: stored, later workers: added, so in worker order).
template <int RP>
__device__ __forceinline__ void p1_reduce(const P1Tile& T, float (&acc)[Cfg<RP>::RSB * RP], int sb, int rn,
                                          float* s_red_w, bool first) {
  constexpr int RSB = Cfg<RP>::RSB;
  float tot;
  const int j = warp_reduce_multi<RSB * RP>(acc, tot);
  constexpr int SH = 5 - (RSB * RP == 1 ? 0 : (RSB * RP == 2 ? 1 : (RSB * RP == 4 ? 2 : (RSB * RP == 8 ? 3 : (RSB * RP == 16 ? 4 : 5)))));
  if ((T.lane & ((1 << SH) - 1)) == 0 && j < rn * RP) {
    float& dst = s_red_w[sb * RP + j];
    dst = first ? tot : dst + tot;
  }
}

// The tile's P rows are complete in s_prow (visible to the CTA): for a layer
// of several segments the row block's last CTA sums the segments' rows (fixed
// order); then P is written and the Gram tail runs.
template <int RP>
__device__ __forceinline__ void p1_rows_done(const StepArgs& a, const LayerDev& L, const P1Tile& T, float* s_prow,
                                             double* s_gram, int* s_flag, unsigned* pub) {
  if (L.s1 > 1) {
    float* pp = a.ppart + L.ppart_off + ((int64_t)T.rb * L.s1 + T.seg) * L.r1 * RP;
    for (int idx = threadIdx.x; idx < T.rcnt * RP; idx += blockDim.x) pp[idx] = s_prow[idx];
    if (!cta_arrive_last(a.counters + L.cnt_off + L.c_rb + T.rb, (unsigned)L.s1, s_flag)) return;
    const float* pb = a.ppart + L.ppart_off + (int64_t)T.rb * L.s1 * L.r1 * RP;
    for (int idx = threadIdx.x; idx < T.rcnt * RP; idx += blockDim.x) {
      float s = 0.f;
      if constexpr (RP <= 4) {
        // loads batched (at r >= 16 this pushes the tensor-core tile's
        // registers into spills)
#pragma unroll 12
        for (int qq = 0; qq < L.s1; ++qq) s += __ldcg(pb + (int64_t)qq * L.r1 * RP + idx);
      } else {
        for (int qq = 0; qq < L.s1; ++qq) s += __ldcg(pb + (int64_t)qq * L.r1 * RP + idx);
      }
      s_prow[idx] = s;
    }
    __syncthreads();
  }
  for (int idx = threadIdx.x; idx < T.rcnt * RP; idx += blockDim.x)
    a.P[L.p_off + (int64_t)T.row0 * RP + idx] = s_prow[idx];
  if (T.ub || a.split) return;  // the unbiased variant sends P as it is; a split step all-reduces it first
  gram_tail<RP>(a, L, T.rb, s_prow, T.rcnt, s_gram, s_flag, pub);
}

// One project tile.  The CTA's warps are split into row groups of
// WG = min(W, warps) warps each; warp v takes the passes (RSB rows) p with
// p % NH == v / WG and the workers v % WG, v % WG + WG, ...  With one warp
// per worker (WG = warps, NH = 1) every warp takes every pass.  Each pass's
// RSB rows of G and B are loaded into registers (streaming loads), then
// used; a warp's lanes load their Q and Q_w' rows straight into registers,
// so the only barrier of a tile is the final sum over the warps of each
// row's group, in worker order.  s_red: warps x R1 x RP floats.
template <int RP>
__device__ __forceinline__ void p1_body(const StepArgs& a, const Tile& t, float* s_red, float* s_prow,
                                        double* s_gram, int* s_flag, unsigned* pub) {
  constexpr int RSB = Cfg<RP>::RSB;
  constexpr int R1 = Cfg<RP>::R1;
  const LayerDev L = a.layers[t.layer];  // by value: stores to B cannot alias it
  const P1Tile T = p1_tile<RP>(a, t, L);
  const int WG = min(a.W, T.nwarps);
  const int NH = T.nwarps / WG;
  const int h = T.warp / WG, wv = T.warp % WG;
  if (h < NH) {
    const float* Pprev = a.Phat + L.p_off + (int64_t)T.row0 * RP;  // previous Phat rows of the tile
    // this lane's 4 Q rows, held in registers for the whole tile
    float qv[4][RP];
    p1_load_q<RP>(a.Qbar + L.q_off, T, false, qv);
    bool first = true;
    for (int w = wv; w < a.W; w += WG) {
      const float* Gw = a.G[w] + L.off + 4 * T.c;
      float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * T.c;
      float qw[4][RP];
      p1_load_q<RP>(a.Qw + (int64_t)w * a.q_total + L.q_off, T, !T.prev, qw);
      for (int sb = h * RSB; sb < T.rcnt; sb += NH * RSB) {
        const int rn = min(RSB, T.rcnt - sb);
        float4 g[RSB], b[RSB];
#pragma unroll
        for (int i = 0; i < RSB; ++i) {
          if (T.act && i < rn) {
            const int64_t o = (int64_t)(T.row0 + sb + i) * L.ld;
            g[i] = __ldcs(reinterpret_cast<const float4*>(Gw + o));
            b[i] = T.ub ? zero4() : __ldcs(reinterpret_cast<const float4*>(Bw + o));
          } else {
            g[i] = zero4();
            b[i] = zero4();
          }
        }
        float acc[RSB * RP];
        p1_rows<RP>(L, T, g, b, sb, rn, Pprev, qv, qw, Bw, acc);
        p1_reduce<RP>(T, acc, sb, rn, s_red + T.warp * R1 * RP, first);
      }
      first = false;
    }
  }
  __syncthreads();
  // P rows: the fixed-order sum over the workers' warps of each row's group
  for (int idx = threadIdx.x; idx < T.rcnt * RP; idx += blockDim.x) {
    const int hh = (idx / RP / RSB) % NH;
    float s = 0.f;
    for (int v = 0; v < WG; ++v) s += s_red[(hh * WG + v) * R1 * RP + idx];
    s_prow[idx] = s;
  }
  __syncthreads();
  p1_rows_done<RP>(a, L, T, s_prow, s_gram, s_flag, pub);
}

template <int RP>
__global__ void __launch_bounds__(32 * Cfg<RP>::P1_WARPS, Cfg<RP>::P1_MINB) p1_kernel(const StepArgs a) {
  constexpr int R1 = Cfg<RP>::R1;
  constexpr int NW = Cfg<RP>::P1_WARPS;
  __shared__ float s_red[NW * R1 * RP];  // per-warp P partials
  __shared__ float s_prow[R1 * RP];
  __shared__ double s_gram[RP * RP];
  __shared__ int s_flag;
  pdl_enter();
  p1_body<RP>(a, a.tiles[blockIdx.x], s_red, s_prow, s_gram, &s_flag, nullptr);
}

// ----------------------------------------------------------------------------
// orthonormalise: Cholesky-QR2, P1 = P R^-1, then X = R2^-1 from P1's Gram
// ----------------------------------------------------------------------------

// One orthonormalise tile: rows chunk * NR .. + NR - 1 of layer L, NR =
// ph_rows(RP), one thread per row (the other threads of the CTA skip the row
// work and only help with the sums).  P1 = P R^-1 by forward substitution in
// float64, rounded to float32 and stored over P.  When the first pass was
// orthogonal enough (the flag gram_finish set), that is the basis: at r >= 8,
// and at r <= 4 when the back-project forms Q_w from Y, the tile also stores
// it as Phat (otherwise, at r <= 4, the back-project stages Phat from P1),
// and it only counts itself done.  Otherwise the tile's rounded
// rows go to shared memory and their Gram matrix (float64, each entry summed
// over the rows in order) to the tile's partial slot.  The partials are
// summed in two levels, each in a fixed order: the last tile of each group
// of kGramGroup tiles sums the group's partials, and the last group sums the
// groups, factors the total (Cholesky, R2) and stores X = R2^-1, so that
// Phat = P1 X.  (One CTA summing every tile's partial took one dependent L2
// round trip per few loads and dominated the phase at r = 32.)  s_r: RP x RP
// + RP doubles; s_p1: NR x RP floats; s_gram: RP x RP doubles.  pub (fused
// step only): the layer's X flag, raised once the layer's tiles are done.
template <int RP>
__device__ __forceinline__ void ph_body(const StepArgs& a, const LayerDev& L, int chunk, double* s_r, float* s_p1,
                                        double* s_gram, int* s_flag, unsigned* pub) {
  constexpr int NG = Cfg<RP>::NG;
  constexpr int NR = ph_rows(RP);
  double* fr = a.rinv + L.rinv_off;
  // the row thread's P row is requested first, with the factor's loads
  const int row = chunk * NR + (int)threadIdx.x;
  const bool valid = threadIdx.x < NR && row < L.n;
  float* prow = a.P + L.p_off + (int64_t)row * RP;
  double x[RP];
#pragma unroll
  for (int k = 0; k < RP; ++k) x[k] = valid ? (double)__ldcg(prow + k) : 0.0;
  for (int e = threadIdx.x; e < RP * RP + RP; e += blockDim.x) s_r[e] = __ldcg(fr + e);
  const bool one_pass = __ldcg(fr + 2 * RP * RP + RP) != 0.0;
  // Phat is stored here at r >= 8, and at r <= 4 when the back-project
  // forms Q_w from Y (it then stages no Phat rows)
  const bool store_phat = one_pass && (RP >= 8 || __ldcg(fr + 2 * RP * RP + RP + 1) != 0.0);
  __syncthreads();
  if (threadIdx.x < NR) {  // whole warps (NR is a multiple of 32)
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      double s = x[k];
#pragma unroll
      for (int j = 0; j < k; ++j) s = fma(-x[j], s_r[j * RP + k], s);
      x[k] = s * s_r[RP * RP + k];
    }
    float xf[RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) xf[k] = (float)x[k];
    if (valid) {
#pragma unroll
      for (int k = 0; k < RP; ++k) prow[k] = xf[k];
      if (store_phat)
#pragma unroll
        for (int k = 0; k < RP; ++k) a.Phat[L.p_off + (int64_t)row * RP + k] = xf[k];
    }
    if (!one_pass)
#pragma unroll
      for (int k = 0; k < RP; ++k) s_p1[threadIdx.x * RP + k] = valid ? xf[k] : 0.f;
  }
  unsigned* cnt = a.counters + L.cnt_off;
  if (one_pass) {
    // the layer is done once every tile has stored its rows (the fused step
    // raises its X flag then; the phase kernels need no count: the
    // back-project waits for the whole grid)
    if (pub && cta_arrive_last(cnt + L.c_ph, (unsigned)L.nph, s_flag) && threadIdx.x == 0) flag_raise(pub, a.epoch);
    return;
  }
  __syncthreads();
  double* gp = a.gram + L.gram_off + (int64_t)(L.nrb + L.g1) * NG;  // the P1 partials: tiles, then groups
  for (int e = threadIdx.x; e < NG; e += blockDim.x) {
    int i, j;
    tri_index(e, RP, i, j);
    double s = 0.0;
    for (int rr = 0; rr < NR; ++rr) s = fma((double)s_p1[rr * RP + i], (double)s_p1[rr * RP + j], s);
    gp[(int64_t)chunk * NG + e] = s;
  }
  const int grp = chunk / kGramGroup;
  const int ngrp = (int)ph_groups(L.nph);
  const int gsz = min(kGramGroup, L.nph - grp * kGramGroup);
  if (!cta_arrive_last(cnt + L.c_phg + grp, (unsigned)gsz, s_flag)) return;
  for (int e = threadIdx.x; e < NG; e += blockDim.x) {
    const double* src = gp + (int64_t)grp * kGramGroup * NG + e;
    double s = 0.0;
#pragma unroll 8
    for (int t = 0; t < gsz; ++t) s += __ldcg(src + (int64_t)t * NG);
    gp[(int64_t)(L.nph + grp) * NG + e] = s;
  }
  if (!cta_arrive_last(cnt + L.c_ph, (unsigned)ngrp, s_flag)) return;
  for (int e = threadIdx.x; e < NG; e += blockDim.x) {
    const double* src = gp + (int64_t)L.nph * NG + e;
    double s = 0.0;
#pragma unroll 8
    for (int g = 0; g < ngrp; ++g) s += __ldcg(src + (int64_t)g * NG);
    int i, j;
    tri_index(e, RP, i, j);
    s_gram[i * RP + j] = s;
    s_gram[j * RP + i] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    warp_cholesky<RP>(s_gram, s_r);  // R2 and 1 / diag R2 (s_r's R is no longer needed)
    __syncwarp();
    warp_tri_inverse<RP>(s_r, fr + RP * RP + RP);
    if (pub) {
      __syncwarp();
      if (threadIdx.x == 0) flag_raise(pub, a.epoch);
    }
  }
}

template <int RP>
__global__ void __launch_bounds__(kPhThreads) ph_kernel(const StepArgs a) {
  static_assert(ph_rows(RP) % 32 == 0 && ph_rows(RP) <= kPhThreads, "the row threads are whole warps of the CTA");
  __shared__ double s_r[RP * RP + RP];
  __shared__ float s_p1[ph_rows(RP) * RP];
  __shared__ double s_gram[RP * RP];
  __shared__ int s_flag;
  __shared__ EarlyTables s_tab;
  stage_tables_early(a, &s_tab, false);
  pdl_enter();
  __syncthreads();
  const LayerDev L = s_tab.L;  // a copy: stores to P cannot alias it
  ph_body<RP>(a, L, s_tab.t.a, s_r, s_p1, s_gram, &s_flag, nullptr);
}

// r >= 8, second pass: Phat rows = P1 X (float64 products, rounded), once per
// row, for the layers whose first pass was not orthogonal enough (the other
// layers' orthonormalise tiles stored Phat already).  The same tiles as the
// orthonormalise phase.
template <int RP>
__global__ void __launch_bounds__(ph_rows(RP)) pf_kernel(const StepArgs a) {
  __shared__ double s_x[RP * RP];
  pdl_enter();
  const Tile t = a.tiles[blockIdx.x];
  const LayerDev L = a.layers[t.layer];
  const double* X = a.rinv + L.rinv_off + RP * RP + RP;
  if (X[RP * RP] != 0.0) return;  // one pass was enough (uniform over the CTA)
  for (int e = threadIdx.x; e < RP * RP; e += blockDim.x) s_x[e] = X[e];
  __syncthreads();
  const int row = t.a * ph_rows(RP) + threadIdx.x;
  if (row >= L.n) return;
  const float* p1 = a.P + L.p_off + (int64_t)row * RP;
  double x[RP];
#pragma unroll
  for (int j = 0; j < RP; ++j) x[j] = (double)p1[j];
  float* out = a.Phat + L.p_off + (int64_t)row * RP;
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    double v = 0.0;
#pragma unroll
    for (int j = 0; j <= k; ++j) v = fma(x[j], s_x[j * RP + k], v);
    out[k] = (float)v;
  }
}

// Split step: the Gram factor of an all-reduced P.  One CTA per project row
// block (segment 0's tile of the project phase): the block's P rows, then
// the same Gram tail the project phase runs.
template <int RP>
__global__ void __launch_bounds__(kGramThreads) gram_kernel(const StepArgs a) {
  __shared__ float s_prow[Cfg<RP>::R1MAX * RP];
  __shared__ double s_gram[RP * RP];
  __shared__ int s_flag;
  pdl_enter();
  const Tile t = a.tiles[blockIdx.x];
  const LayerDev L = a.layers[t.layer];
  const int row0 = t.a * L.r1;
  const int rcnt = min(L.r1, L.n - row0);
  for (int idx = threadIdx.x; idx < rcnt * RP; idx += blockDim.x)
    s_prow[idx] = __ldcg(a.P + L.p_off + (int64_t)row0 * RP + idx);
  __syncthreads();
  gram_tail<RP>(a, L, t.a, s_prow, rcnt, s_gram, &s_flag, nullptr);
}

// ----------------------------------------------------------------------------
// back-project: partial Q_w = M_w^T Phat over a row tile; segment finalise
// ----------------------------------------------------------------------------
template <int RP>
__device__ void qbar_segment(const StepArgs& a, const LayerDev& L, int seg, int* s_flag, unsigned* pub);

// pub (fused step only): the segment's Qbar flag, raised once Qbar is stored.
template <int RP>
__device__ void qf_segment_worker(const StepArgs& a, const LayerDev& L, int seg, int w, int* s_flag, unsigned* pub) {
  const int col0 = seg * kSeg * 4;
  const int col1 = min(L.ld, col0 + kSeg * 4);
  const int n4 = (col1 - col0) * RP / 4;  // float4 of the segment's ld x RP slice
  const int64_t e0 = (int64_t)col0 * RP;
  const int64_t wstride = (int64_t)L.ld * RP;
  const int64_t tstride = (int64_t)a.W * wstride;  // from one row tile to the next
  const float* parts = a.qpart + L.qpart_off + (int64_t)w * wstride + e0;
  float* qw = a.Qw + (int64_t)w * a.q_total + L.q_off + e0;
  for (int q = threadIdx.x; q < n4; q += blockDim.x) {
    float4 s = zero4();
    int rt = 0;
    for (; rt + 4 <= L.t3r; rt += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(reinterpret_cast<const float4*>(parts + (rt + u) * tstride) + q);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        s.x += v[u].x;
        s.y += v[u].y;
        s.z += v[u].z;
        s.w += v[u].w;
      }
    }
    for (; rt < L.t3r; ++rt) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(parts + rt * tstride) + q);
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    reinterpret_cast<float4*>(qw)[q] = s;
  }
  qbar_segment<RP>(a, L, seg, s_flag, pub);
}

// The CTA has stored Q_w of one worker over segment seg: the segment's last
// worker forms Qbar = qbar_scale * sum_w Q_w (worker order).
template <int RP>
__device__ void qbar_segment(const StepArgs& a, const LayerDev& L, int seg, int* s_flag, unsigned* pub) {
  const int col0 = seg * kSeg * 4;
  const int col1 = min(L.ld, col0 + kSeg * 4);
  const int n4 = (col1 - col0) * RP / 4;
  const int64_t e0 = (int64_t)col0 * RP;
  if (!cta_arrive_last(a.counters + L.cnt_off + L.c_qs + seg, (unsigned)a.W, s_flag)) return;
  const float invw = a.qbar_scale;
  for (int q = threadIdx.x; q < n4; q += blockDim.x) {
    float4 s = zero4();
    for (int v = 0; v < a.W; ++v) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(a.Qw + (int64_t)v * a.q_total + L.q_off + e0) + q);
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    reinterpret_cast<float4*>(a.Qbar + L.q_off + e0)[q] = make_float4(s.x * invw, s.y * invw, s.z * invw, s.w * invw);
  }
  if (pub) {
    __syncthreads();
    if (threadIdx.x == 0) flag_raise(pub, a.epoch);
  }
}

// One-pass back-project of worker w over segment seg: Y_w = the sum of the
// layer's Y partial slots (float64; the first half of the slots summed by
// threads 0..127, the second by threads 128..255, each in slot order, then
// first + second), Q_w = Y_w R^-1 (float64, rounded), then Qbar as in the
// two-pass form.  A CTA of 256 threads; s_x: RP x RP doubles; s_half:
// 128 x RP doubles.
template <int RP>
__device__ void qy_segment_worker(const StepArgs& a, const LayerDev& L, int seg, int w, double* s_x, double* s_half,
                                  int* s_flag) {
  const double* ri = a.rinv + L.rinv_off + RP * RP + RP;
  for (int e = threadIdx.x; e < RP * RP; e += blockDim.x) s_x[e] = __ldg(ri + e);
  const int col0 = seg * kSeg * 4;
  const int col1 = min(L.ld, col0 + kSeg * 4);
  const int c = col0 + (int)(threadIdx.x & 127);
  const int h = (int)(threadIdx.x >> 7);
  const int mid = (L.nys + 1) / 2;
  const int g0 = h ? mid : 0, g1 = h ? L.nys : mid;
  const int64_t gstride = (int64_t)a.W * L.ld * RP;  // from one slot to the next
  double y[RP];
#pragma unroll
  for (int k = 0; k < RP; ++k) y[k] = 0.0;
  if (c < col1) {
    const float* src = a.ypart + L.y_off + (int64_t)w * L.ld * RP + (int64_t)c * RP;
#pragma unroll 8
    for (int g = g0; g < g1; ++g) {
      float v[RP];
      if constexpr (RP == 4) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(src + g * gstride));
        v[0] = x.x;
        v[1] = x.y;
        v[2] = x.z;
        v[3] = x.w;
      } else if constexpr (RP == 2) {
        const float2 x = __ldcs(reinterpret_cast<const float2*>(src + g * gstride));
        v[0] = x.x;
        v[1] = x.y;
      } else {
#pragma unroll
        for (int k = 0; k < RP; ++k) v[k] = __ldcs(src + g * gstride + k);
      }
#pragma unroll
      for (int k = 0; k < RP; ++k) y[k] += (double)v[k];
    }
  }
  if (h)
#pragma unroll
    for (int k = 0; k < RP; ++k) s_half[(threadIdx.x & 127) * RP + k] = y[k];
  __syncthreads();
  if (!h && c < col1) {
    float* qw = a.Qw + (int64_t)w * a.q_total + L.q_off;
#pragma unroll
    for (int k = 0; k < RP; ++k) y[k] += s_half[threadIdx.x * RP + k];
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      double q = 0.0;
#pragma unroll
      for (int j = 0; j <= k; ++j) q = fma(y[j], s_x[j * RP + k], q);
      qw[(int64_t)c * RP + k] = (float)q;
    }
  }
  qbar_segment<RP>(a, L, seg, s_flag, nullptr);
}

// Back-project: rank slices per row group (warps that read the same rows),
// and its dynamic shared memory (the cross-warp reduction), in bytes.
constexpr int p3_slices(int rp) { return rp >= 32 ? 2 : 1; }
constexpr size_t p3_dyn_bytes(int rp) { return (size_t)(kP3Threads / 32 / p3_slices(rp)) * 32 * 4 * rp * sizeof(float); }


// One back-project tile (kP3Threads threads) of layer L, UNR rows per warp
// group.
// FUSED: the tile runs inside the fused step, where B, P1 and X were written
// by other CTAs of the same launch, so they are read through L2 only
// (ld.global.cg; an L1 line of this SM could be stale); pub is then the
// segment's Qbar flag.  s_ph: warps x UNR x RH floats; s_x: RP x RP doubles;
// s_red: p3_dyn_bytes(RP) bytes.
template <int RP, int UNR, bool FUSED>
__device__ __forceinline__ void p3_body(const StepArgs& a, const Tile& t, const LayerDev& L, float* s_ph, double* s_x,
                                        float* s_red, int* s_flag, unsigned* pub) {
  constexpr int NW = kP3Threads / 32;
  // r = 32: the ranks are split over warp pairs that read the same rows (the
  // second read hits in cache), so a warp holds 4 x RP / 2 accumulators and
  // two CTAs fit on an SM instead of one
  constexpr int HS = p3_slices(RP);  // rank slices
  constexpr int RH = RP / HS;        // ranks per warp
  constexpr int NG = NW / HS;        // row groups in flight
  static_assert(p3_dyn_bytes(RP) >= (size_t)NW * UNR * RP * sizeof(float), "s_red holds every warp's P1 rows");
  const int rt = t.a, seg = t.b, w = t.c;
  if (!FUSED && RP <= 4 && a.ypath && __ldg(a.rinv + L.rinv_off + 2 * RP * RP + RP + 1) != 0.0) {
    // the project phase formed Y_w = M_w^T P: one tile per (segment, worker)
    // forms Q_w from it, and no tile reads M
    static_assert(p3_dyn_bytes(RP) >= 128 * RP * sizeof(double), "s_red holds the second half's sums");
    if (rt == 0) qy_segment_worker<RP>(a, L, seg, w, s_x, reinterpret_cast<double*>(s_red), s_flag);
    return;
  }
  const int row0 = rt * L.r3;
  const int nrows = min(L.r3, L.n - row0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hs = warp % HS, grp = warp / HS;
  const int c = seg * kSeg + lane;
  const bool act = c < L.F;
  const float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * c;
  // r <= 4 (and the fused step): the Phat rows are formed here from P1 (and
  // X after a second pass; float64 products of RP terms) as they are staged,
  // and one tile per row tile stores them.  r >= 8: the orthonormalise phase
  // stored Phat.
  constexpr bool kForm = FUSED || RP <= 4;
  const float* P1 = (kForm ? a.P : a.Phat) + L.p_off + (int64_t)row0 * RP;
  float* Pout = (kForm && seg == 0 && w == 0) ? a.Phat + L.p_off + (int64_t)row0 * RP : nullptr;
  const double* X = a.rinv + L.rinv_off + RP * RP + RP;
  float4 bv[UNR];
  auto load_rows = [&](int i0) {
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const float4* src = reinterpret_cast<const float4*>(Bw + (int64_t)(row0 + i0 + u) * L.ld);
      bv[u] = (act && i0 + u < nrows) ? (FUSED ? __ldcg(src) : (HS > 1 ? __ldg(src) : __ldcs(src))) : zero4();
    }
  };
  // r <= 4: the first group's rows go out before the X flag is known (they
  // need only the layer record), so the flag's load overlaps them; outside
  // the fused step so does the lane's value of the group's P1 rows, which
  // is Phat when one pass was enough (UNR x RH <= 32: one value a lane)
  constexpr bool kEarly = !FUSED && RP <= 4;
  static_assert(!kEarly || UNR * RH <= 32, "one early P1 value per lane");
  if (kForm) load_rows(grp * UNR);
  float p_early = 0.f;
  if (kEarly && grp * UNR < nrows && lane < min(UNR, nrows - grp * UNR) * RH)
    p_early = __ldg(P1 + (int64_t)(grp * UNR + lane / RH) * RP + hs * RH + lane % RH);
  const bool ident = !kForm || (FUSED ? __ldcg(X + RP * RP) : __ldg(X + RP * RP)) != 0.0;
  if (!ident) {
    for (int e = threadIdx.x; e < RP * RP; e += blockDim.x) s_x[e] = FUSED ? __ldcg(X + e) : __ldg(X + e);
    __syncthreads();
  }
  float* s_mine = s_ph + warp * UNR * RH;
  float* s_p1 = s_red + warp * UNR * RP;  // this warp's P1 rows (before the final reduction)
  float acc[4][RH];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < RH; ++k) acc[j][k] = 0.f;
  // row groups of UNR rows interleaved over the NG groups; each warp stages
  // its own slice of the group's Phat rows (warp barriers only) while the
  // group's B rows are in flight
  for (int i0 = grp * UNR; i0 < nrows; i0 += NG * UNR) {
    const int nr = min(UNR, nrows - i0);
    __syncwarp();  // the previous group's rows are no longer read
    if (!kForm || i0 != grp * UNR) load_rows(i0);
    if (!ident) {
      // Phat = P1 X (j ascending): the group's P1 rows (all ranks), then the
      // product
      for (int e = lane; e < nr * RP; e += 32)
        s_p1[e] = FUSED ? __ldcg(P1 + (int64_t)i0 * RP + e) : __ldg(P1 + (int64_t)i0 * RP + e);
      __syncwarp();
      for (int e = lane; e < nr * RH; e += 32) {
        const int u = e / RH, k = hs * RH + e % RH;
        // float64: when P was nearly rank deficient, X has large entries and
        // the terms cancel (X was formed from these rounded P1 values, so
        // the exact product is orthonormal)
        double v = 0.0;
#pragma unroll 8
        for (int j = 0; j < RP; ++j) v = fma((double)s_p1[u * RP + j], s_x[j * RP + k], v);
        s_mine[e] = (float)v;
        if (Pout) Pout[(int64_t)(i0 + u) * RP + k] = (float)v;
      }
    } else {  // Phat = P1
      for (int e = lane; e < nr * RH; e += 32) {
        const int64_t o = (int64_t)(i0 + e / RH) * RP + hs * RH + e % RH;
        const float v = (kEarly && i0 == grp * UNR) ? p_early : (FUSED ? __ldcg(P1 + o) : __ldg(P1 + o));
        s_mine[e] = v;
        if (Pout) Pout[o] = v;
      }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (i0 + u < nrows) {
#pragma unroll
        for (int k = 0; k < RH; ++k) {
          const float p = s_mine[u * RH + k];
          acc[0][k] = fmaf(bv[u].x, p, acc[0][k]);
          acc[1][k] = fmaf(bv[u].y, p, acc[1][k]);
          acc[2][k] = fmaf(bv[u].z, p, acc[2][k]);
          acc[3][k] = fmaf(bv[u].w, p, acc[3][k]);
        }
      }
    }
  }
  // fixed-order reduction over the row groups (s_red held the warps' P1 rows)
  __syncthreads();
  float* mine = s_red + (grp * 32 + lane) * 4 * RP + hs * RH;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < RH; ++k) mine[j * RP + k] = acc[j][k];
  __syncthreads();
  // a layer of one row tile: the tile's sum is Q_w itself (the same value
  // the sum over one partial gives), stored without the partial's round
  // trip through L2
  const bool direct = L.t3r == 1;
  {
    float* part = direct ? a.Qw + (int64_t)w * a.q_total + L.q_off
                         : a.qpart + L.qpart_off + ((int64_t)rt * a.W + w) * L.ld * RP;
    const int ncol4 = min(kSeg, L.F - seg * kSeg);
    for (int idx = threadIdx.x; idx < ncol4 * 4 * RP; idx += blockDim.x) {
      const int ln = idx / (4 * RP), jk = idx % (4 * RP);
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < NG; ++v) s += s_red[(v * 32 + ln) * 4 * RP + jk];
      part[(int64_t)(seg * kSeg + ln) * 4 * RP + jk] = s;
    }
  }
  if (direct)
    qbar_segment<RP>(a, L, seg, s_flag, pub);
  else if (cta_arrive_last(a.counters + L.cnt_off + L.c_p3 + seg * a.W + w, (unsigned)L.t3r, s_flag))
    qf_segment_worker<RP>(a, L, seg, w, s_flag, pub);
}

template <int RP>
__global__ void __launch_bounds__(kP3Threads, Cfg<RP>::P3_MINB) p3_kernel(const StepArgs a) {
  constexpr int UNR = Cfg<RP>::UNR3;
  constexpr int RH = RP / p3_slices(RP);
  __shared__ float s_ph[(kP3Threads / 32) * UNR * RH];  // each warp's Phat values of its current group
  __shared__ double s_x[RP * RP];                       // X = R2^-1 (when it is not the identity)
  extern __shared__ __align__(16) float s_red[];        // the cross-warp reduction; first each warp's P1 rows
  __shared__ int s_flag;
  if constexpr (RP >= 16) {
    // two CTAs per SM of 27 or more waves: the early staging's barrier costs
    // more than the first wave's round trips it saves
    pdl_enter();
    const Tile t = a.tiles[blockIdx.x];
    const LayerDev L = a.layers[t.layer];  // by value: stores to B cannot alias it
    p3_body<RP, UNR, false>(a, t, L, s_ph, s_x, s_red, &s_flag, nullptr);
  } else {
    __shared__ EarlyTables s_tab;
    stage_tables_early(a, &s_tab, false);
    pdl_enter();
    __syncthreads();
    const Tile t = s_tab.t;
    const LayerDev L = s_tab.L;  // a copy: stores to B cannot alias it
    p3_body<RP, UNR, false>(a, t, L, s_ph, s_x, s_red, &s_flag, nullptr);
  }
}

// ----------------------------------------------------------------------------
// decompress: rows of Phat Qbar^T; vector layers: worker mean
// ----------------------------------------------------------------------------

// Momentum-SGD update of one element by the decompressed u:
// mom <- beta mom + u, x <- x - lr (u + mom).
__device__ __forceinline__ void momentum1(float& x, float& mom, float u, float lr, float beta) {
  mom = fmaf(beta, mom, u);
  x = fmaf(-lr, u + mom, x);
}

// The same for the float4 at p of X and Mom; elements at or past `valid`
// (row padding) are left as they are.
__device__ __forceinline__ void momentum4(float* X, float* Mom, int64_t p, float4 u, int valid, float lr,
                                          float beta) {
  float4 x = __ldcs(reinterpret_cast<const float4*>(X + p));
  float4 m = __ldcs(reinterpret_cast<const float4*>(Mom + p));
  momentum1(x.x, m.x, u.x, lr, beta);
  if (valid > 1) momentum1(x.y, m.y, u.y, lr, beta);
  if (valid > 2) momentum1(x.z, m.z, u.z, lr, beta);
  if (valid > 3) momentum1(x.w, m.w, u.w, lr, beta);
  __stcs(reinterpret_cast<float4*>(X + p), x);
  __stcs(reinterpret_cast<float4*>(Mom + p), m);
}
// One decompress tile (kUThreads threads): of layer L, or (t.c == 1) of the
// vector layers, L unused.  FUSED: Phat and Qbar were written by other CTAs
// of the same launch and are read through L2 only.  s_ph: RU x RP floats.
template <int RP, bool FUSED>
__device__ __forceinline__ void u_body(const StepArgs& a, const Tile& t, const LayerDev& L, float* s_ph) {
  constexpr int RU = Cfg<RP>::RU;
  if (t.c == 1) {  // vector layer: U = mean_w G_w
    const VecDev V = a.vecs[t.layer];
    const int base = t.a * kVChunk;
    const int end = min(V.n, base + kVChunk);
    for (int i = base + (int)threadIdx.x; i < end; i += blockDim.x) {
      float s = 0.f;
      for (int w = 0; w < a.W; ++w) s += __ldcs(a.G[w] + V.off + i);
      const float u = s / (float)a.W;
      if (a.U) a.U[V.off + i] = u;
      if (a.X) {
        float x = a.X[V.off + i], mom = a.Mom[V.off + i];
        momentum1(x, mom, u, a.lr, a.beta);
        a.X[V.off + i] = x;
        a.Mom[V.off + i] = mom;
      }
    }
    return;
  }
  const int row0 = t.a * L.ru, seg = t.b;
  const int rcnt = min(L.ru, L.n - row0);
  const float* Psrc = (a.unbiased ? a.P : a.Phat) + L.p_off + (int64_t)row0 * RP;
  const int lane = threadIdx.x & 31, sub = threadIdx.x >> 5;  // 8 rows in flight per pass
  const int c = seg * kSeg + lane;
  // the lane's Qbar rows are requested with the Phat rows, before the barrier
  float qv[4][RP];
  if (c < L.F) {
    const float* qs = a.Qbar + L.q_off + (int64_t)(4 * c) * RP;
    float* flat = &qv[0][0];
    if constexpr (RP % 4 == 0) {
      const float4* qb = reinterpret_cast<const float4*>(qs);
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const float4 v = FUSED ? __ldcg(qb + i) : __ldg(qb + i);
        flat[4 * i] = v.x;
        flat[4 * i + 1] = v.y;
        flat[4 * i + 2] = v.z;
        flat[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4 * RP; ++i) flat[i] = FUSED ? __ldcg(qs + i) : __ldg(qs + i);
    }
  }
  for (int i = threadIdx.x; i < rcnt * RP; i += blockDim.x) s_ph[i] = FUSED ? __ldcg(Psrc + i) : __ldg(Psrc + i);
  __syncthreads();
  if (c >= L.F) return;
  const int valid = (c == L.F - 1) ? L.tail : 4;
  const int64_t col = L.off + 4 * c;
#pragma unroll 4
  for (int r = sub; r < rcnt; r += kUThreads / 32) {
    float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      const float p = s_ph[r * RP + k];
      u0 = fmaf(p, qv[0][k], u0);
      u1 = fmaf(p, qv[1][k], u1);
      u2 = fmaf(p, qv[2][k], u2);
      u3 = fmaf(p, qv[3][k], u3);
    }
    if (a.unbiased) {
      u0 *= a.u_scale;
      u1 *= a.u_scale;
      u2 *= a.u_scale;
      u3 *= a.u_scale;
    }
    const int64_t pos = col + (int64_t)(row0 + r) * L.ld;
    if (a.U) __stcs(reinterpret_cast<float4*>(a.U + pos), make_float4(u0, u1, u2, u3));
    if (a.X) momentum4(a.X, a.Mom, pos, make_float4(u0, u1, u2, u3), valid, a.lr, a.beta);
  }
}

template <int RP>
__global__ void __launch_bounds__(kUThreads) u_kernel(const StepArgs a) {
  __shared__ float s_ph[Cfg<RP>::RU * RP];
  __shared__ EarlyTables s_tab;
  stage_tables_early(a, &s_tab, true);
  pdl_enter();
  __syncthreads();
  const Tile t = s_tab.t;
  const LayerDev L = s_tab.L;  // a copy (matrix tiles only): stores to U cannot alias it
  u_body<RP, false>(a, t, L, s_ph);
}

// ----------------------------------------------------------------------------
// r >= 8: register-tiled project and decompress
// ----------------------------------------------------------------------------
//
// At r >= 8 the lane-per-4-columns project and decompress kernels would
// hold 8 r floats of Q rows per lane; these kernels instead spread the
// r-wide dot products so that each value loaded from shared memory feeds
// several fused multiply-adds.  (The back-project kernel serves every rank.)

constexpr int kTThreads = 256;  // threads of a tiled project CTA: 32 rows x 8 column groups

// Project, r >= 8.  A CTA owns up to 32 rows x one segment (128 columns) and
// loops over the workers.  Thread (row i = tid / 8, column group cg = tid % 8)
// owns the float4 columns cg, cg + 8, cg + 16, cg + 24 of its row (16
// columns; each of the 8 threads of a row reads a different 16 bytes, so the
// loads of a warp are coalesced and the shared-memory reads conflict-free).
// Per worker: E = B - Phat' Q_w'^T for its 16 elements (fmaf chains, k
// ascending, as in the error read-back kernel), M = G + E stored to B and
// added to the thread's running sum over the workers.  After the last
// worker, its share of the P row, sum_c (sum_w M_w)[i][c] Q[c][k]: one r-wide
// product per tile instead of one per worker (P is linear in M).  The 8
// column groups of a row are summed with a butterfly over their 8 lanes.
// Q and Q_w' are staged transposed ([k][column]) so a thread reads its 4
// float4 columns at fixed k.
// The tiled project kernel's G and B float4 of worker w: row i of the tile,
// float4 columns c40 + 8 v (zeros past the row or the layer; no B in the
// unbiased variant).
__device__ __forceinline__ void p1t_load_gb(const StepArgs& a, const LayerDev& L, const P1Tile& T, int w, int i,
                                            int c40, bool row_ok, float4 (&gv)[4], float4 (&bv)[4]) {
  const float4* G4 = reinterpret_cast<const float4*>(a.G[w] + L.off + (int64_t)(T.row0 + i) * L.ld);
  const float4* B4 = reinterpret_cast<const float4*>(a.B + (int64_t)w * a.total + L.off + (int64_t)(T.row0 + i) * L.ld);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int c4 = c40 + 8 * v;
    gv[v] = zero4();
    bv[v] = zero4();
    if (row_ok && c4 < L.F) {
      gv[v] = __ldcs(G4 + c4);
      if (!T.ub) bv[v] = __ldcs(B4 + c4);
    }
  }
}

template <int RP>
__global__ void __launch_bounds__(kTThreads, 2) p1t_kernel(const StepArgs a) {
  constexpr int TR = 32;
  constexpr int SC = kSeg * 4;  // columns of a segment
  constexpr int SCP = kP1TRow;  // their row stride in shared memory (padded: the staging stores hit 4-way, not 32-way)
  static_assert(Cfg<RP>::R1 == TR && TR * 8 == kTThreads, "the tiled project kernel covers 32 rows, 8 threads each");
  extern __shared__ __align__(16) float s_t[];
  float* s_qT = s_t;               // Q rows of the segment, transposed: [RP][SCP]
  float* s_qwT = s_qT + RP * SCP;  // Q_w' rows of the current worker, transposed: [RP][SCP]
  float* s_pp = s_qwT + RP * SCP;  // previous Phat rows of the tile: [TR][RP]
  __shared__ float s_prow[TR * RP];
  __shared__ double s_gram[RP * RP];
  __shared__ int s_flag;
  pdl_enter();
  const Tile t = a.tiles[blockIdx.x];
  const LayerDev L = a.layers[t.layer];  // by value
  const P1Tile T = p1_tile<RP>(a, t, L);
  const int i = threadIdx.x >> 3, cg = threadIdx.x & 7;
  const bool row_ok = i < T.rcnt;
  const int c40 = T.seg * kSeg + cg;  // float4 column of v = 0; v-th is c40 + 8 v
  const int64_t q0 = L.q_off + (int64_t)T.seg * SC * RP;
  const int segcols = min(SC, L.ld - T.seg * SC);
  // staging: rank fastest, so consecutive threads load consecutive words
  // (the rows are m x RP in memory) and store down a padded column
  for (int e = threadIdx.x; e < RP * SC; e += blockDim.x) {
    const int c = e / RP, k = e - c * RP;
    s_qT[k * SCP + c] = c < segcols ? __ldg(a.Qbar + q0 + e) : 0.f;
  }
  for (int e = threadIdx.x; e < TR * RP; e += blockDim.x)
    s_pp[e] = (T.prev && e < T.rcnt * RP) ? __ldg(a.Phat + L.p_off + (int64_t)T.row0 * RP + e) : 0.f;
  float msum[16];  // sum over the workers of the thread's 16 M values
  // each worker's Q_w' values are loaded one worker ahead (NQ per thread) and
  // stored into shared memory after the barrier, so their latency hides
  // behind the previous worker's arithmetic
  constexpr int NQ = RP * SC / kTThreads;
  static_assert(NQ * kTThreads == RP * SC, "whole staging rows per thread");
  float qv[NQ];
  auto fetch_qw = [&](int wk) {
    const float* qw = a.Qw + (int64_t)wk * a.q_total + q0;
#pragma unroll
    for (int u = 0; u < NQ; ++u) {
      const int e = threadIdx.x + u * kTThreads;
      qv[u] = (e / RP) < segcols ? __ldg(qw + e) : 0.f;
    }
  };
  if (T.prev) fetch_qw(0);
  // below r = 32 the registers allow G and B to be loaded one worker ahead
  constexpr bool kAhead = RP <= 16;
  float4 gn[4], bn[4];
  if (kAhead) p1t_load_gb(a, L, T, 0, i, c40, row_ok, gn, bn);
  for (int w = 0; w < a.W; ++w) {
    // this worker's G and B first: their loads are in flight during the staging
    float* Bw = a.B + (int64_t)w * a.total + L.off + (int64_t)(T.row0 + i) * L.ld;
    float4 gc[4], bc[4];
    if (kAhead) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        gc[v] = gn[v];
        bc[v] = bn[v];
      }
      if (w + 1 < a.W) p1t_load_gb(a, L, T, w + 1, i, c40, row_ok, gn, bn);
    } else {
      p1t_load_gb(a, L, T, w, i, c40, row_ok, gc, bc);
    }
    float g[16], m[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      g[4 * v] = gc[v].x; g[4 * v + 1] = gc[v].y; g[4 * v + 2] = gc[v].z; g[4 * v + 3] = gc[v].w;
      m[4 * v] = bc[v].x; m[4 * v + 1] = bc[v].y; m[4 * v + 2] = bc[v].z; m[4 * v + 3] = bc[v].w;
    }
    __syncthreads();  // the previous worker's Q_w' rows are no longer read
    if (T.prev) {
#pragma unroll
      for (int u = 0; u < NQ; ++u) {
        const int e = threadIdx.x + u * kTThreads;
        const int c = e / RP, k = e - c * RP;
        s_qwT[k * SCP + c] = qv[u];
      }
    }
    __syncthreads();
    if (T.prev && w + 1 < a.W) fetch_qw(w + 1);
    if (T.prev) {
#pragma unroll 4
      for (int k = 0; k < RP; ++k) {
        const float p = s_pp[i * RP + k];
        const float4* qk = reinterpret_cast<const float4*>(s_qwT + k * SCP) + cg;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 q = qk[8 * v];
          m[4 * v] = fmaf(-p, q.x, m[4 * v]);
          m[4 * v + 1] = fmaf(-p, q.y, m[4 * v + 1]);
          m[4 * v + 2] = fmaf(-p, q.z, m[4 * v + 2]);
          m[4 * v + 3] = fmaf(-p, q.w, m[4 * v + 3]);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int c4 = c40 + 8 * v;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int col = 4 * c4 + x;
        m[4 * v + x] = (col < L.m) ? g[4 * v + x] + m[4 * v + x] : 0.f;
      }
      if (row_ok && c4 < L.F && !T.ub)
        reinterpret_cast<float4*>(Bw)[c4] = make_float4(m[4 * v], m[4 * v + 1], m[4 * v + 2], m[4 * v + 3]);
    }
    // the workers' M summed in order: P = (sum_w M_w) Q needs one product
    // per tile, not one per worker
#pragma unroll
    for (int x = 0; x < 16; ++x) msum[x] = (w == 0) ? m[x] : msum[x] + m[x];
  }
  // P partial: for each rank, the thread's 16 columns in order
  float pacc[RP];
#pragma unroll 4
  for (int k = 0; k < RP; ++k) {
    const float4* qk = reinterpret_cast<const float4*>(s_qT + k * SCP) + cg;
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 q = qk[8 * v];
      acc = fmaf(msum[4 * v], q.x, acc);
      acc = fmaf(msum[4 * v + 1], q.y, acc);
      acc = fmaf(msum[4 * v + 2], q.z, acc);
      acc = fmaf(msum[4 * v + 3], q.w, acc);
    }
    pacc[k] = acc;
  }
  // sum the 8 column groups of each row (lanes 8 (i % 4) + cg): a fixed
  // butterfly that leaves lane cg with ranks [base, base + RP / 8)
  {
    int base = 0;
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      const int o = 4 >> l;             // lane bit 2, 1, 0 of cg
      const int half = RP >> (l + 1);   // values still held / 2
      const bool up = (cg & o) != 0;
#pragma unroll
      for (int x = 0; x < half; ++x) {
        const float send = up ? pacc[x] : pacc[x + half];
        const float keep = up ? pacc[x + half] : pacc[x];
        pacc[x] = keep + __shfl_xor_sync(kFull, send, o);
      }
      if (up) base += half;
    }
    if (row_ok)
#pragma unroll
      for (int x = 0; x < RP / 8; ++x) s_prow[i * RP + base + x] = pacc[x];
  }
  __syncthreads();
  p1_rows_done<RP>(a, L, T, s_prow, s_gram, &s_flag, nullptr);
}

// Decompress, r >= 8: thread = one column of the segment (its Q rows, RP
// floats, in registers), rows walked with the Phat rows broadcast from
// shared memory; vector layers as in u_kernel.
template <int RP>
__global__ void __launch_bounds__(kSeg * 4) ut_kernel(const StepArgs a) {
  constexpr int RU = Cfg<RP>::RU;
  __shared__ __align__(16) float s_ph[RU * RP];
  __shared__ EarlyTables s_tab;
  stage_tables_early(a, &s_tab, true);
  pdl_enter();
  __syncthreads();
  const Tile t = s_tab.t;
  if (t.c == 1) {  // vector layer: U = mean_w G_w
    const VecDev V = a.vecs[t.layer];
    const int base = t.a * kVChunk;
    const int end = min(V.n, base + kVChunk);
    for (int i = base + (int)threadIdx.x; i < end; i += blockDim.x) {
      float s = 0.f;
      for (int w = 0; w < a.W; ++w) s += __ldcs(a.G[w] + V.off + i);
      const float u = s / (float)a.W;
      if (a.U) a.U[V.off + i] = u;
      if (a.X) {
        float x = a.X[V.off + i], mom = a.Mom[V.off + i];
        momentum1(x, mom, u, a.lr, a.beta);
        a.X[V.off + i] = x;
        a.Mom[V.off + i] = mom;
      }
    }
    return;
  }
  const LayerDev L = s_tab.L;  // a copy: stores to U cannot alias it
  const int row0 = t.a * L.ru, seg = t.b;
  const int rcnt = min(L.ru, L.n - row0);
  const float* Psrc = a.unbiased ? a.P : a.Phat;
  for (int i = threadIdx.x; i < rcnt * RP; i += blockDim.x) s_ph[i] = __ldg(Psrc + L.p_off + (int64_t)row0 * RP + i);
  __syncthreads();
  const int col = seg * kSeg * 4 + threadIdx.x;
  if (col >= L.ld) return;
  float q[RP];
  {
    const float4* qs = reinterpret_cast<const float4*>(a.Qbar + L.q_off + (int64_t)col * RP);
#pragma unroll
    for (int k4 = 0; k4 < RP / 4; ++k4) {
      const float4 v = __ldg(qs + k4);
      q[4 * k4] = v.x; q[4 * k4 + 1] = v.y; q[4 * k4 + 2] = v.z; q[4 * k4 + 3] = v.w;
    }
  }
  const bool valid = col < L.m;
  for (int r = 0; r < rcnt; ++r) {
    const float4* ph = reinterpret_cast<const float4*>(s_ph + r * RP);
    float u = 0.f;
#pragma unroll
    for (int k4 = 0; k4 < RP / 4; ++k4) {
      const float4 p = ph[k4];
      u = fmaf(p.x, q[4 * k4], u);
      u = fmaf(p.y, q[4 * k4 + 1], u);
      u = fmaf(p.z, q[4 * k4 + 2], u);
      u = fmaf(p.w, q[4 * k4 + 3], u);
    }
    if (a.unbiased) u *= a.u_scale;
    const int64_t pos = L.off + (int64_t)(row0 + r) * L.ld + col;
    if (a.U) __stcs(a.U + pos, u);
    if (a.X && valid) {
      float x = a.X[pos], mom = a.Mom[pos];
      momentum1(x, mom, u, a.lr, a.beta);
      a.X[pos] = x;
      a.Mom[pos] = mom;
    }
  }
}

// ----------------------------------------------------------------------------
// side kernels: Q initialisation, error read-back
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

#ifdef PSGD_SIDE_KERNELS
// Q of matrix layer blockIdx.y: N(0,1) from splitmix64 keyed by (seed, layer
// position) + Box-Muller, rounded to float32, row-major m x r inside the
// ld x RP buffer (padding stays as set by the caller: zero).
__global__ void q_init_kernel(float* Qbar, const LayerDev* layers, int rank, int RP, uint64_t seed) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ull;
  const LayerDev L = layers[blockIdx.y];
  const uint64_t key = splitmix64_mix(seed + (uint64_t)(L.index + 1) * gamma);
  const int64_t total = (int64_t)L.m * rank;
  const int64_t pairs = (total + 1) / 2;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < pairs;
       t += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t x1 = splitmix64_mix(key + (uint64_t)(2 * t + 1) * gamma);
    const uint64_t x2 = splitmix64_mix(key + (uint64_t)(2 * t + 2) * gamma);
    const double u1 = (double)((x1 >> 11) + 1ull) * (1.0 / 9007199254740992.0);
    const double u2 = (double)((x2 >> 11) + 1ull) * (1.0 / 9007199254740992.0);
    const double rad = sqrt(-2.0 * log(u1));
    const double ang = 2.0 * CUDART_PI * u2;
    const int64_t e0 = 2 * t, e1 = 2 * t + 1;
    Qbar[L.q_off + (e0 / rank) * RP + (e0 % rank)] = (float)(rad * cos(ang));
    if (e1 < total) Qbar[L.q_off + (e1 / rank) * RP + (e1 % rank)] = (float)(rad * sin(ang));
  }
}
#endif  // PSGD_SIDE_KERNELS

// E = B - Phat Q_w^T of one layer and worker, dense n x m.  The k loop runs
// in the same order with the same fused multiply-adds as the project phase's
// correction, so the values are exactly the ones the next step adds to its
// gradient.
template <int RP>
__global__ void error_kernel(float* E, const float* B, const float* Phat, const float* Qw, int n, int m, int ld) {
  const int64_t total = (int64_t)n * m;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / m, j = idx % m;
    float e = B[i * ld + j];
#pragma unroll
    for (int k = 0; k < RP; ++k) e = fmaf(-Phat[i * RP + k], Qw[j * RP + k], e);
    E[idx] = e;
  }
}

}  // namespace psgd
