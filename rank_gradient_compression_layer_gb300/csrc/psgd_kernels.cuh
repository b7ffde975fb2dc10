// Device code of the PowerSGD compression step for sm_103a.
//
// One persistent kernel runs a whole step.  Its CTAs take work items from an
// in-order queue; an item may wait (bounded) on a per-layer flag that an
// EARLIER item publishes, so the queue always drains.  Per matrix layer:
//
//   P1  (row tiles)  M_w = G_w + (B_w - Phat' Q_w'^T)   B holds M of the last
//                    step, so the bracket is the error E_w; store B_w <- M_w;
//                    P rows = (sum_w M_w) Q; partial Gram P^T P of the tile.
//                    The last tile of the layer sums the Gram (fixed order,
//                    float64), factors it (Cholesky, float64) and publishes
//                    R^-1:  Phat = P R^-1 is the Gram-Schmidt basis of P.
//   PH  (row tiles)  Phat rows = P rows R^-1 (float64 -> float32).
//   P3  (row tile x segment x worker)  partial Q_w = M_w^T Phat over the tile's
//                    rows; the last tile of a segment sums the partials (fixed
//                    order) into Q_w and Qbar = mean_w Q_w.
//   U   (row tiles)  U rows = Phat Qbar^T (only when an update is requested).
//   V   vector layers: U = mean_w G_w.
//
// The error buffer is never written as such: E_w = B_w - Phat Q_w^T is rebuilt
// on the fly by the next step's P1 (r FMAs per element), which saves a full
// read+write pass over every error buffer.
//
// All reductions run in a fixed order, so a step is bit-reproducible.  Data
// written by another CTA during the same launch is read with ld.global.cg
// (L2), never through L1.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "psgd_internal.h"

namespace psgd {

template <int RP>
struct Cfg {
  static constexpr int NG = RP * (RP + 1) / 2;         // Gram entries (upper triangle)
  static constexpr int KC = RP < 8 ? RP : 8;           // rank chunk held in registers
  static constexpr int RS1 = RP <= 4 ? 8 : (RP == 8 ? 4 : (RP == 16 ? 2 : 1));  // P1 rows per pair
  static constexpr int RSU = RP <= 8 ? 8 : 4;          // U rows per pair
  static constexpr int UNR3 = 8;                       // P3 rows in flight per warp
};

constexpr int kVChunk = 4096;  // vector elements per V item

// ----------------------------------------------------------------------------
// memory helpers
// ----------------------------------------------------------------------------

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ float f4get(const float4& v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
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

// ----------------------------------------------------------------------------
// cross-CTA synchronisation (bounded)
// ----------------------------------------------------------------------------

// Thread 0 only.  Polls *flag until it holds `epoch`; gives up after `limit`
// polls (records a timeout in ctl->status) or as soon as another CTA has
// recorded an error.  Returns true when the flag was seen.
static __device__ __noinline__ bool wait_flag(const unsigned* flag, unsigned epoch, Ctl* ctl, int64_t limit,
                                       int where) {
  for (int64_t it = 0;; ++it) {
    if (ld_acquire_u32(flag) == epoch) return true;
    if (*(volatile int*)&ctl->status != 0) return false;
    if (it >= limit) {
      if (atomicCAS(&ctl->status, 0, kDevTimeout) == 0) ctl->where = where;
      return false;
    }
    __nanosleep(128);
  }
}

// All threads: returns whether the flag was seen.
__device__ __forceinline__ bool cta_wait(const unsigned* flag, unsigned epoch, Ctl* ctl, int64_t limit,
                                         int where, int* s_int) {
  if (threadIdx.x == 0) *s_int = wait_flag(flag, epoch, ctl, limit, where) ? 1 : 0;
  __syncthreads();
  const bool ok = *s_int != 0;
  __syncthreads();
  return ok;
}

// All threads: make this CTA's global writes visible, count one arrival on
// *cnt, and return true (in every thread) when this was arrival number
// `total`.  The last arriver resets the counter for the next launch and may
// then read everything the other arrivers wrote (with .cg loads).
__device__ __forceinline__ bool arrive_last(unsigned* cnt, unsigned total, int* s_int) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atom_add_acq_rel(cnt, 1u);
    const bool last = (old == total - 1);
    if (last) *cnt = 0u;
    *s_int = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *s_int != 0;
  __syncthreads();
  return last;
}

// All threads: publish `epoch` in *flag after this CTA's writes.
__device__ __forceinline__ void publish(unsigned* flag, unsigned epoch) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) st_release_u32(flag, epoch);
}

// ----------------------------------------------------------------------------
// Gram-Schmidt coefficients from the Gram matrix (float64, one thread)
// ----------------------------------------------------------------------------
//
// A = P^T P = R^T R with R upper triangular, diag > 0: R is the R factor of
// Gram-Schmidt on the columns of P, and Phat = P R^-1.  A pivot that is not
// positive marks a column whose remainder vanished: its row of R and its
// column of R^-1 are zero, so the matching column of Phat is zero.
template <int RP>
__device__ void cholesky_inverse(const double* A, double* R, double* Ri) {
  bool deg[RP];
  for (int i = 0; i < RP * RP; ++i) R[i] = 0.0;
  for (int j = 0; j < RP; ++j) {
    double d = A[j * RP + j];
    for (int k = 0; k < j; ++k) d -= R[k * RP + j] * R[k * RP + j];
    if (!(d > 0.0)) {
      deg[j] = true;
      continue;
    }
    deg[j] = false;
    const double rjj = sqrt(d);
    R[j * RP + j] = rjj;
    for (int i = j + 1; i < RP; ++i) {
      double s = A[j * RP + i];
      for (int k = 0; k < j; ++k) s -= R[k * RP + j] * R[k * RP + i];
      R[j * RP + i] = s / rjj;
    }
  }
  for (int i = 0; i < RP * RP; ++i) Ri[i] = 0.0;
  for (int k = 0; k < RP; ++k) {
    if (deg[k]) continue;
    Ri[k * RP + k] = 1.0 / R[k * RP + k];
    for (int a = k - 1; a >= 0; --a) {
      if (deg[a]) continue;
      double s = 0.0;
      for (int b = a + 1; b <= k; ++b) s += R[a * RP + b] * Ri[b * RP + k];
      Ri[a * RP + k] = -s / R[a * RP + a];
    }
  }
}

// Last P1 group of a layer: sum the group Grams, factor, publish R^-1.
template <int RP>
__device__ void gram_finalize(const StepArgs& a, const LayerDev& L, float* smem) {
  constexpr int NG = Cfg<RP>::NG;
  double* A = reinterpret_cast<double*>(smem);
  double* R = A + RP * RP;
  double* Ri = R + RP * RP;
  const double* gg = a.gram + L.gram_off + (int64_t)L.t1 * NG;
  for (int e = threadIdx.x; e < NG; e += kThreads) {
    double s = 0.0;
    for (int g = 0; g < L.g1; ++g) s += __ldcg(gg + (int64_t)g * NG + e);
    int i, j;
    tri_index(e, RP, i, j);
    A[i * RP + j] = s;
    A[j * RP + i] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) cholesky_inverse<RP>(A, R, Ri);
  __syncthreads();
  for (int e = threadIdx.x; e < RP * RP; e += kThreads) a.rinv[L.rinv_off + e] = Ri[e];
  publish(&a.flags[L.flag_off + 0], a.epoch);
}

// ----------------------------------------------------------------------------
// P1: error add, B <- M, P = (sum_w M_w) Q, Gram partial
// ----------------------------------------------------------------------------
template <int RP>
__device__ void p1_tile(const StepArgs& a, const LayerDev& L, int tile, float* smem, int* s_int) {
  constexpr int RS = Cfg<RP>::RS1;
  constexpr int KC = Cfg<RP>::KC;
  constexpr int NG = Cfg<RP>::NG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row0 = tile * L.r1;
  const int nrows = min(L.r1, L.n - row0);
  float* s_pprev = smem;                    // r1 x RP : Phat of the last step
  float* s_psum = s_pprev + L.r1 * RP;      // kWarps x r1 x RP
  for (int i = tid; i < L.r1 * RP; i += kThreads)
    s_pprev[i] = (a.has_prev && i < nrows * RP) ? __ldcg(a.Phat + L.p_off + (int64_t)row0 * RP + i) : 0.f;
  for (int i = tid; i < kWarps * L.r1 * RP; i += kThreads) s_psum[i] = 0.f;
  __syncthreads();

  const int npairs = L.S * L.rho1;
  for (int pr = warp; pr < npairs; pr += kWarps) {
    const int seg = pr % L.S, sb = pr / L.S;
    const int rlo = sb * RS;
    const int rcnt = min(RS, nrows - rlo);
    if (rcnt <= 0) continue;  // warp-uniform
    const int c = seg * kSeg + lane;
    const bool act = c < L.F;
    const bool tailc = act && (c == L.F - 1) && (L.tail < 4);
    float ms[RS][4];
#pragma unroll
    for (int i = 0; i < RS; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) ms[i][j] = 0.f;

    for (int w = 0; w < a.W; ++w) {
      const float* Gw = a.G[w] + L.off + 4 * c;
      float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * c;
      float4 g[RS], b[RS];
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        if (act && i < rcnt) {
          const int64_t o = (int64_t)(row0 + rlo + i) * L.ld;
          g[i] = __ldcs(reinterpret_cast<const float4*>(Gw + o));
          b[i] = __ldcg(reinterpret_cast<const float4*>(Bw + o));
        } else {
          g[i] = zero4();
          b[i] = zero4();
        }
      }
      float e[RS][4];
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        e[i][0] = b[i].x;
        e[i][1] = b[i].y;
        e[i][2] = b[i].z;
        e[i][3] = b[i].w;
      }
      if (a.has_prev) {
        // E_w = B_w - Phat' Q_w'^T, k in ascending order (the same chain as
        // the error read-back kernel)
        const float* Qw = a.Qw + (int64_t)w * a.q_total + L.q_off + (int64_t)(4 * c) * RP;
#pragma unroll
        for (int k0 = 0; k0 < RP; k0 += KC) {
          float qw[4][KC];
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int kk = 0; kk < KC; ++kk) qw[j][kk] = act ? __ldcg(Qw + j * RP + k0 + kk) : 0.f;
#pragma unroll
          for (int i = 0; i < RS; ++i) {
#pragma unroll
            for (int kk = 0; kk < KC; ++kk) {
              const float p = s_pprev[(rlo + i) * RP + k0 + kk];
#pragma unroll
              for (int j = 0; j < 4; ++j) e[i][j] = fmaf(-p, qw[j][kk], e[i][j]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        if (act && i < rcnt) {
          float mv[4];
          mv[0] = f4get(g[i], 0) + e[i][0];
          mv[1] = f4get(g[i], 1) + e[i][1];
          mv[2] = f4get(g[i], 2) + e[i][2];
          mv[3] = f4get(g[i], 3) + e[i][3];
          if (tailc) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j >= L.tail) mv[j] = 0.f;
          }
          *reinterpret_cast<float4*>(Bw + (int64_t)(row0 + rlo + i) * L.ld) =
              make_float4(mv[0], mv[1], mv[2], mv[3]);
#pragma unroll
          for (int j = 0; j < 4; ++j) ms[i][j] += mv[j];
        }
      }
    }

    // project the worker sum onto the warm-start Q
    const float* Qb = a.Qbar + L.q_off + (int64_t)(4 * c) * RP;
#pragma unroll
    for (int k0 = 0; k0 < RP; k0 += KC) {
      float qv[4][KC];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int kk = 0; kk < KC; ++kk) qv[j][kk] = act ? __ldcg(Qb + j * RP + k0 + kk) : 0.f;
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        if (i < rcnt) {  // warp-uniform
#pragma unroll
          for (int kk = 0; kk < KC; ++kk) {
            float s = ms[i][0] * qv[0][kk];
            s = fmaf(ms[i][1], qv[1][kk], s);
            s = fmaf(ms[i][2], qv[2][kk], s);
            s = fmaf(ms[i][3], qv[3][kk], s);
            s = warp_sum(s);
            if (lane == 0) s_psum[(warp * L.r1 + rlo + i) * RP + k0 + kk] += s;
          }
        }
      }
    }
  }
  __syncthreads();

  // P rows of the tile: fixed-order sum over warps
  float* s_prow = s_pprev;
  for (int idx = tid; idx < nrows * RP; idx += kThreads) {
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < kWarps; ++v) s += s_psum[v * L.r1 * RP + idx];
    s_prow[idx] = s;
    a.P[L.p_off + (int64_t)row0 * RP + idx] = s;
  }
  __syncthreads();

  // Gram partial of the tile (float64; products of floats are exact)
  double* gp = a.gram + L.gram_off + (int64_t)tile * NG;
  for (int e = tid; e < NG; e += kThreads) {
    int i, j;
    tri_index(e, RP, i, j);
    double s = 0.0;
    for (int rr = 0; rr < nrows; ++rr) s = fma((double)s_prow[rr * RP + i], (double)s_prow[rr * RP + j], s);
    gp[e] = s;
  }

  const int grp = tile / kGramGroup;
  const int gsz = min(kGramGroup, L.t1 - grp * kGramGroup);
  unsigned* cnt = a.counters + L.cnt_off;
  if (arrive_last(cnt + 1 + grp, (unsigned)gsz, s_int)) {
    double* gg = a.gram + L.gram_off + (int64_t)(L.t1 + grp) * NG;
    const double* parts = a.gram + L.gram_off + (int64_t)grp * kGramGroup * NG;
    for (int e = tid; e < NG; e += kThreads) {
      double s = 0.0;
      for (int t = 0; t < gsz; ++t) s += __ldcg(parts + (int64_t)t * NG + e);
      gg[e] = s;
    }
    if (arrive_last(cnt, (unsigned)L.g1, s_int)) gram_finalize<RP>(a, L, smem);
  }
}

// ----------------------------------------------------------------------------
// PH: Phat rows = P rows R^-1 (float64)
// ----------------------------------------------------------------------------
template <int RP>
__device__ void ph_tile(const StepArgs& a, const LayerDev& L, int tile, float* smem, int* s_int) {
  double* s_ri = reinterpret_cast<double*>(smem);
  for (int e = threadIdx.x; e < RP * RP; e += kThreads) s_ri[e] = __ldcg(a.rinv + L.rinv_off + e);
  __syncthreads();
  const int row = tile * L.rph + threadIdx.x;
  if (threadIdx.x < L.rph && row < L.n) {
    double p[RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) p[k] = (double)__ldcg(a.P + L.p_off + (int64_t)row * RP + k);
    float* out = a.Phat + L.p_off + (int64_t)row * RP;
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      double s = 0.0;
#pragma unroll
      for (int j = 0; j <= k; ++j) s = fma(p[j], s_ri[j * RP + k], s);
      out[k] = (float)s;
    }
  }
  unsigned* cnt = a.counters + L.cnt_off + 1 + L.g1;
  if (arrive_last(cnt, (unsigned)L.tph, s_int)) publish(&a.flags[L.flag_off + 1], a.epoch);
}

// ----------------------------------------------------------------------------
// P3: partial Q_w = M_w^T Phat over r3 rows of one segment; segment finalise
// ----------------------------------------------------------------------------
template <int RP>
__device__ void qf_segment(const StepArgs& a, const LayerDev& L, int seg, int* s_int) {
  const int col0 = seg * kSeg * 4;
  const int col1 = min(L.ld, col0 + kSeg * 4);
  const int nel = (col1 - col0) * RP;
  const int64_t wstride = (int64_t)L.ld * RP;
  const float* parts = a.qpart + L.qpart_off;
  for (int idx = threadIdx.x; idx < nel; idx += kThreads) {
    const int64_t e = (int64_t)col0 * RP + idx;
    float qb = 0.f;
    for (int w = 0; w < a.W; ++w) {
      float s = 0.f;
      for (int rt = 0; rt < L.t3r; ++rt) s += __ldcg(parts + ((int64_t)rt * a.W + w) * wstride + e);
      a.Qw[(int64_t)w * a.q_total + L.q_off + e] = s;
      qb += s;
    }
    a.Qbar[L.q_off + e] = qb / (float)a.W;
  }
  unsigned* cnt = a.counters + L.cnt_off + 2 + L.g1;
  if (arrive_last(cnt, (unsigned)L.S, s_int)) publish(&a.flags[L.flag_off + 2], a.epoch);
}

template <int RP>
__device__ void p3_tile(const StepArgs& a, const LayerDev& L, int rt, int segw, float* smem, int* s_int) {
  constexpr int UNR = Cfg<RP>::UNR3;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = segw / a.W, w = segw % a.W;
  const int row0 = rt * L.r3;
  const int nrows = min(L.r3, L.n - row0);
  // warps split the tile's rows into contiguous ranges
  const int per = (nrows + kWarps - 1) / kWarps;
  const int wr0 = min(nrows, warp * per);
  const int wr1 = min(nrows, wr0 + per);
  const int c = seg * kSeg + lane;
  const bool act = c < L.F;
  float* s_ph = smem + warp * 32 * RP;                  // per-warp Phat staging (32 rows)
  float* s_red = smem + kWarps * 32 * RP;               // kWarps x 32 lanes x 4 x RP
  const float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * c;
  float acc[4][RP];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < RP; ++k) acc[j][k] = 0.f;

  for (int r0 = wr0; r0 < wr1; r0 += 32) {
    const int rn = min(32, wr1 - r0);
    __syncwarp();
    for (int idx = lane; idx < rn * RP; idx += 32)
      s_ph[idx] = __ldcg(a.Phat + L.p_off + (int64_t)(row0 + r0) * RP + idx);
    __syncwarp();
    for (int i0 = 0; i0 < rn; i0 += UNR) {
      float4 bv[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        bv[u] = (act && i0 + u < rn)
                    ? __ldcs(reinterpret_cast<const float4*>(Bw + (int64_t)(row0 + r0 + i0 + u) * L.ld))
                    : zero4();
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (i0 + u < rn) {  // warp-uniform
#pragma unroll
          for (int k = 0; k < RP; ++k) {
            const float p = s_ph[(i0 + u) * RP + k];
            acc[0][k] = fmaf(bv[u].x, p, acc[0][k]);
            acc[1][k] = fmaf(bv[u].y, p, acc[1][k]);
            acc[2][k] = fmaf(bv[u].z, p, acc[2][k]);
            acc[3][k] = fmaf(bv[u].w, p, acc[3][k]);
          }
        }
      }
    }
  }
  // fixed-order reduction over the warps (row ranges ascend with the warp index)
  float* mine = s_red + (warp * 32 + lane) * 4 * RP;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < RP; ++k) mine[j * RP + k] = acc[j][k];
  __syncthreads();
  {
    float* part = a.qpart + L.qpart_off + ((int64_t)rt * a.W + w) * L.ld * RP;
    const int ncol4 = min(kSeg, L.F - seg * kSeg);
    for (int idx = tid; idx < ncol4 * 4 * RP; idx += kThreads) {
      const int ln = idx / (4 * RP), jk = idx % (4 * RP);
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < kWarps; ++v) s += s_red[(v * 32 + ln) * 4 * RP + jk];
      part[(int64_t)(seg * kSeg + ln) * 4 * RP + jk] = s;
    }
  }
  unsigned* cnt = a.counters + L.cnt_off + 3 + L.g1 + seg;
  if (arrive_last(cnt, (unsigned)(L.t3r * a.W), s_int)) qf_segment<RP>(a, L, seg, s_int);
}

// ----------------------------------------------------------------------------
// U: rows of Phat Qbar^T
// ----------------------------------------------------------------------------
template <int RP>
__device__ void u_tile(const StepArgs& a, const LayerDev& L, int tile, float* smem) {
  constexpr int RS = Cfg<RP>::RSU;
  constexpr int KC = Cfg<RP>::KC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row0 = tile * L.ru;
  const int nrows = min(L.ru, L.n - row0);
  float* s_ph = smem;
  for (int i = tid; i < nrows * RP; i += kThreads) s_ph[i] = __ldcg(a.Phat + L.p_off + (int64_t)row0 * RP + i);
  __syncthreads();
  const int npairs = L.S * L.rhou;
  for (int pr = warp; pr < npairs; pr += kWarps) {
    const int seg = pr % L.S, sb = pr / L.S;
    const int rlo = sb * RS;
    const int rcnt = min(RS, nrows - rlo);
    if (rcnt <= 0) continue;
    const int c = seg * kSeg + lane;
    const bool act = c < L.F;
    const float* Qb = a.Qbar + L.q_off + (int64_t)(4 * c) * RP;
    float u[RS][4];
#pragma unroll
    for (int i = 0; i < RS; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) u[i][j] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < RP; k0 += KC) {
      float qv[4][KC];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int kk = 0; kk < KC; ++kk) qv[j][kk] = act ? __ldcg(Qb + j * RP + k0 + kk) : 0.f;
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        if (i < rcnt) {
#pragma unroll
          for (int kk = 0; kk < KC; ++kk) {
            const float p = s_ph[(rlo + i) * RP + k0 + kk];
#pragma unroll
            for (int j = 0; j < 4; ++j) u[i][j] = fmaf(p, qv[j][kk], u[i][j]);
          }
        }
      }
    }
    if (act) {
      float* Ub = a.U + L.off + 4 * c;
#pragma unroll
      for (int i = 0; i < RS; ++i)
        if (i < rcnt)
          __stcs(reinterpret_cast<float4*>(Ub + (int64_t)(row0 + rlo + i) * L.ld),
                 make_float4(u[i][0], u[i][1], u[i][2], u[i][3]));
    }
  }
}

// ----------------------------------------------------------------------------
// V: worker mean of a vector layer
// ----------------------------------------------------------------------------
__device__ __forceinline__ void v_tile(const StepArgs& a, const VecDev& V, int tile) {
  const int base = tile * kVChunk;
  const int end = min(V.n, base + kVChunk);
  for (int i = base + (int)threadIdx.x; i < end; i += kThreads) {
    float s = 0.f;
    for (int w = 0; w < a.W; ++w) s += __ldcs(a.G[w] + V.off + i);
    a.U[V.off + i] = s / (float)a.W;
  }
}

// ----------------------------------------------------------------------------
// the persistent step kernel
// ----------------------------------------------------------------------------
template <int RP>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const StepArgs a) {
  extern __shared__ __align__(16) float smem[];
  __shared__ int s_int[2];
  for (;;) {
    if (threadIdx.x == 0) {
      unsigned it = atomicAdd(&a.ctl->next, 1u);
      if (*(volatile int*)&a.ctl->status != 0) it = 0x7fffffffu;
      s_int[0] = (int)min(it, 0x7fffffffu);
    }
    __syncthreads();
    const int it = s_int[0];
    __syncthreads();
    if (it >= a.num_items) break;
    const Item item = a.items[it];
    if (item.kind == kItemV) {
      if (a.U != nullptr) v_tile(a, a.vecs[item.layer], item.a);
    } else {
      const LayerDev& L = a.layers[item.layer];
      switch (item.kind) {
        case kItemP1:
          p1_tile<RP>(a, L, item.a, smem, s_int + 1);
          break;
        case kItemPH:
          if (cta_wait(&a.flags[L.flag_off + 0], a.epoch, a.ctl, a.spin_limit, it, s_int + 1))
            ph_tile<RP>(a, L, item.a, smem, s_int + 1);
          break;
        case kItemP3:
          if (cta_wait(&a.flags[L.flag_off + 1], a.epoch, a.ctl, a.spin_limit, it, s_int + 1))
            p3_tile<RP>(a, L, item.a, item.b, smem, s_int + 1);
          break;
        case kItemU:
          if (a.U != nullptr &&
              cta_wait(&a.flags[L.flag_off + 2], a.epoch, a.ctl, a.spin_limit, it, s_int + 1))
            u_tile<RP>(a, L, item.a, smem);
          break;
        default:
          break;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned e = atomicAdd(&a.ctl->exited, 1u);
    if (e == gridDim.x - 1) {
      a.ctl->next = 0u;
      a.ctl->exited = 0u;
    }
  }
}

// Dynamic shared memory the step kernel needs for one context.
template <int RP>
size_t step_smem_bytes(int max_r1, int max_ru) {
  size_t p1 = (size_t)(1 + kWarps) * max_r1 * RP * sizeof(float);
  size_t gf = (size_t)3 * RP * RP * sizeof(double);
  size_t p3 = (size_t)kWarps * 32 * RP * sizeof(float) + (size_t)kWarps * 32 * 4 * RP * sizeof(float);
  size_t u = (size_t)max_ru * RP * sizeof(float);
  size_t s = p1;
  if (gf > s) s = gf;
  if (p3 > s) s = p3;
  if (u > s) s = u;
  return s;
}

// ----------------------------------------------------------------------------
// side kernels: Q initialisation, error read-back, wait self-test
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
// in the same order with the same fused multiply-adds as the P1 correction,
// so the values are exactly the ones the next step adds to its gradient.
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

#ifdef PSGD_SIDE_KERNELS
__global__ void wait_selftest_kernel(unsigned* flag, Ctl* ctl, int64_t limit) {
  __shared__ int s_int;
  cta_wait(flag, 1u, ctl, limit, 0, &s_int);
}
#endif  // PSGD_SIDE_KERNELS

}  // namespace psgd
