// Device code of the PowerSGD compression step for sm_103a.
//
// One persistent kernel runs a whole step.  Every WARP is an independent
// worker: it claims work items from an in-order queue (one atomic per item,
// issued one item ahead) and processes each item alone, so no CTA barrier
// ever stalls the streaming warps and the load balances at warp granularity.
// An item may wait (bounded) on a per-layer flag that an EARLIER item
// publishes, so the queue always drains.  Per matrix layer:
//
//   P1  (r1 rows x NF4 float4 columns)  M_w = G_w + (B_w - Phat' Q_w'^T): B holds M
//       of the last step, so the bracket is the error E_w; store B_w <- M_w;
//       partial P rows = (sum_w M_w) Q.  The warp that completes a row block
//       writes its P rows and their Gram partial P^T P (float64); the warp
//       that completes the layer sums the Gram (fixed order), factors it
//       A = R^T R (Cholesky, float64, warp-parallel) and publishes R:
//       Phat = P R^-1 is the Gram-Schmidt basis of P.
//   PH  (32 rows)  Phat rows: forward substitution Phat R = P (float64).
//   P3  (r3 rows x one segment x one worker)  partial Q_w = M_w^T Phat; the
//       warp that completes a segment sums the partials (fixed order) into
//       Q_w and Qbar = mean_w Q_w.
//   U   (rsu rows x gsu segments)  U rows = Phat Qbar^T (when requested).
//   V   vector layers: U = mean_w G_w.
//
// The error buffer is never written as such: E_w = B_w - Phat Q_w^T is rebuilt
// on the fly by the next step's P1 (r FMAs per element), which saves a full
// read+write pass over every error buffer.
//
// All reductions run in a fixed order, so a step is bit-reproducible.  Data
// written by another warp during the same launch is read with ld.global.cg
// (L2), never through L1.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "psgd_internal.h"

namespace psgd {

template <int RP>
struct Cfg {
  static constexpr int NG = RP * (RP + 1) / 2;                 // Gram entries (upper triangle)
  // P1 items: R1 rows x NF4 float4 columns, streamed in stages of RS1 rows of one worker
  static constexpr int RS1 = RP <= 4 ? 4 : (RP == 8 ? 2 : 1);
  static constexpr int R1 = 16;
  static constexpr int NF4 = RP <= 8 ? 32 : 256 / RP;
  static constexpr int QSPAN = NF4 * 16 * RP;                 // bytes of a Q span (4 NF4 rows of RP floats)
  static constexpr int P1_SLOT = 2 * RS1 * NF4 * 16 + QSPAN;  // G rows, B rows, Q_w span
  static constexpr int HDR = QSPAN + R1 * RP * 4;             // per item: Qbar span, previous Phat rows
  // P3 items: r3 rows x one segment x one worker, in stages of R3C rows
  static constexpr int R3C = 8;
  static constexpr int P3_SLOT = R3C * kSeg * 16 + R3C * RP * 4 + 16;
  // U items: RSU rows x GSU segments (one Qbar span staged in one slot)
  static constexpr int RSU = RP <= 8 ? 8 : 4;
  static constexpr int SLOT_A = P1_SLOT > P3_SLOT ? P1_SLOT : P3_SLOT;
  static constexpr int SLOT = ((SLOT_A + 127) / 128) * 128;
  static constexpr int GSU = SLOT / (kSeg * 16 * RP) > 0 ? SLOT / (kSeg * 16 * RP) : 1;
  static constexpr int NST = 4;                               // ring slots per warp
  // per-warp shared memory: NST mbarriers, NST slots, 2 item headers, P rows, U Phat rows
  static constexpr int BAR_BYTES = 64;
  static constexpr int PROW_BYTES = R1 * RP * 4 > RSU * RP * 4 ? R1 * RP * 4 : RSU * RP * 4;
  static constexpr int WSM_BYTES = BAR_BYTES + NST * SLOT + 2 * ((HDR + 15) / 16) * 16 + ((PROW_BYTES + 15) / 16) * 16;
  static constexpr int MINB = 1;                              // the shared memory decides residency
};

constexpr int kVChunk = 1024;  // vector elements per V item
constexpr unsigned kFull = 0xffffffffu;

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

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned smid() {
  unsigned r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
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

// Load K consecutive floats through L2 (vectorised when K allows).
template <int K>
__device__ __forceinline__ void ld_row_cg(float* dst, const float* src) {
  if constexpr (K % 4 == 0) {
#pragma unroll
    for (int k = 0; k < K; k += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + k));
      dst[k] = v.x;
      dst[k + 1] = v.y;
      dst[k + 2] = v.z;
      dst[k + 3] = v.w;
    }
  } else if constexpr (K == 2) {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
    dst[0] = v.x;
    dst[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) dst[k] = __ldcg(src + k);
  }
}

// ----------------------------------------------------------------------------
// cross-warp synchronisation (bounded)
// ----------------------------------------------------------------------------

// Lane 0 only.  Polls *flag until it holds `epoch`; gives up after `limit`
// polls (records a timeout in ctl->status) or as soon as another warp has
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
    __nanosleep(64);
  }
}

// Whole warp: returns whether the flag was seen.
__device__ __forceinline__ bool warp_wait(const unsigned* flag, unsigned epoch, Ctl* ctl, int64_t limit, int where) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_flag(flag, epoch, ctl, limit, where) ? 1 : 0;
  ok = __shfl_sync(kFull, ok, 0);
  return ok != 0;
}

// Whole warp: make the warp's global writes visible, count one arrival on
// *cnt, and return true (in every lane) when this was arrival number
// `total`.  The last arriver resets the counter for the next launch and may
// then read everything the other arrivers wrote (with .cg loads).
__device__ __forceinline__ bool warp_arrive_last(unsigned* cnt, unsigned total) {
  __threadfence();
  __syncwarp();
  unsigned old = 0;
  if ((threadIdx.x & 31) == 0) old = atom_add_acq_rel(cnt, 1u);
  old = __shfl_sync(kFull, old, 0);
  const bool last = (old == total - 1);
  if (last && (threadIdx.x & 31) == 0) *cnt = 0u;
  __syncwarp();
  return last;
}

// Whole warp: publish `epoch` in *flag after the warp's writes.
__device__ __forceinline__ void warp_publish(unsigned* flag, unsigned epoch) {
  __threadfence();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) st_release_u32(flag, epoch);
  __syncwarp();
}

// ----------------------------------------------------------------------------
// bulk copies (TMA) into per-warp shared-memory stages
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// One arrival that also announces `bytes` of copies to wait for.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  uint64_t state;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
               : "=l"(state)
               : "r"(smem_u32(bar)), "r"(bytes)
               : "memory");
  (void)state;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Global -> shared bulk copy (16-byte aligned, size a multiple of 16) that
// completes `bytes` on the mbarrier; `policy` is an L2 eviction policy.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Order this thread's earlier generic-proxy accesses before its later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Whole warp: wait (bounded) until the copies announced on `bar` for the phase
// with parity `parity` have landed.  On a timeout it records the error, waits
// once more (bounded) for the copies in flight and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, Ctl* ctl, int64_t limit, int where) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) {
    for (int64_t it = 0; it < limit; ++it) {
      if (mbar_try_wait(bar, parity)) {
        ok = 1;
        break;
      }
    }
    if (!ok) {
      if (atomicCAS(&ctl->status, 0, kDevTimeout) == 0) ctl->where = where;
      for (int64_t it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) break;
    }
  }
  ok = __shfl_sync(kFull, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Per-warp pipeline state that lives across items.  Every staged item kind
// streams its bulk copies through one ring of NST slots; `head` counts the
// stages issued and `tail` the stages consumed (slot = count % NST), and bit s
// of `phase` is the parity the next wait on slot s expects.
struct WarpPipe {
  uint64_t* bar;      // NST mbarriers
  char* ring;         // NST slots
  char* hdr;          // 2 P1 item headers
  float* prow;        // P rows of a P1 item / Phat rows of a U item
  int slot_bytes, hdr_bytes;
  unsigned phase;
  unsigned head, tail;
  int pre_item;       // P1 item whose first `pre_count` stages are already issued, or -1
  int pre_count;
  int hb;             // header of the next P1 item
  uint64_t pol_first;
};

__device__ __forceinline__ char* slot_ptr(const WarpPipe& wp, unsigned count, int nst) {
  return wp.ring + (count % nst) * wp.slot_bytes;
}

// Whole warp: wait for the oldest issued stage and return its slot index.
template <int NST>
__device__ __forceinline__ bool ring_pop(WarpPipe& wp, Ctl* ctl, int64_t limit, int where, int& slot) {
  slot = (int)(wp.tail % NST);
  if (!mbar_wait(wp.bar + slot, (wp.phase >> slot) & 1u, ctl, limit, where)) return false;
  wp.phase ^= 1u << slot;
  return true;
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
// and 1/diag(R) to `out`.
template <int RP>
__device__ void warp_cholesky(const double* A, double* out) {
  const int lane = threadIdx.x & 31;
  double a[RP];
#pragma unroll
  for (int i = 0; i < RP; ++i) a[i] = (lane < RP) ? __ldcg(A + i * RP + lane) : 0.0;
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

// ----------------------------------------------------------------------------
// P1: error add, B <- M, P = (sum_w M_w) Q, Gram partial, Gram finalize
// ----------------------------------------------------------------------------

template <int RP>
__device__ void gram_tail(const StepArgs& a, const LayerDev& L, int rb, const float* prow, int nrows) {
  constexpr int NG = Cfg<RP>::NG;
  const int lane = threadIdx.x & 31;
  unsigned* cnt = a.counters + L.cnt_off;
  double* gp = a.gram + L.gram_off;
  for (int e = lane; e < NG; e += 32) {
    int i, j;
    tri_index(e, RP, i, j);
    double s = 0.0;
    for (int rr = 0; rr < nrows; ++rr) s = fma((double)prow[rr * RP + i], (double)prow[rr * RP + j], s);
    gp[(int64_t)rb * NG + e] = s;
  }
  const int grp = rb / kGramGroup;
  const int gsz = min(kGramGroup, L.nrb - grp * kGramGroup);
  if (!warp_arrive_last(cnt + L.c_grp + grp, (unsigned)gsz)) return;
  for (int e = lane; e < NG; e += 32) {
    double s = 0.0;
    for (int t = 0; t < gsz; ++t) s += __ldcg(gp + (int64_t)(grp * kGramGroup + t) * NG + e);
    gp[(int64_t)(L.nrb + grp) * NG + e] = s;
  }
  if (!warp_arrive_last(cnt + L.c_gram, (unsigned)L.g1)) return;
  // the whole Gram, fixed order over groups, into scratch after R and 1/diag
  double* A = a.rinv + L.rinv_off + RP * RP + RP;
  for (int e = lane; e < NG; e += 32) {
    double s = 0.0;
    for (int g = 0; g < L.g1; ++g) s += __ldcg(gp + (int64_t)(L.nrb + g) * NG + e);
    int i, j;
    tri_index(e, RP, i, j);
    A[i * RP + j] = s;
    A[j * RP + i] = s;
  }
  __threadfence();
  __syncwarp();
  warp_cholesky<RP>(A, a.rinv + L.rinv_off);
  warp_publish(&a.flags[L.flag_off + 0], a.epoch);
}

struct P1Geo {
  int row0, rcnt, f0, nf4, nsb;
};

template <int RP>
__device__ __forceinline__ P1Geo p1_geo(const LayerDev& L, int rb, int sg) {
  P1Geo g;
  g.row0 = rb * Cfg<RP>::R1;
  g.rcnt = min(Cfg<RP>::R1, L.n - g.row0);
  g.f0 = sg * Cfg<RP>::NF4;
  g.nf4 = min(Cfg<RP>::NF4, L.F - g.f0);
  g.nsb = (g.rcnt + Cfg<RP>::RS1 - 1) / Cfg<RP>::RS1;
  return g;
}

// Issue stage s (sub-block s / W, worker s % W) of a P1 item into the ring
// slot of count wp.head; stage 0 also brings the item header (Qbar span and
// the previous Phat rows) into header buffer hb.
template <int RP>
__device__ void p1_issue(const StepArgs& a, const LayerDev& L, const P1Geo& g, int s, int hb, WarpPipe& wp) {
  constexpr int RS1 = Cfg<RP>::RS1;
  constexpr int NF4 = Cfg<RP>::NF4;
  constexpr int NST = Cfg<RP>::NST;
  const int lane = threadIdx.x & 31;
  const int slot = (int)(wp.head % NST);
  char* sl = wp.ring + slot * wp.slot_bytes;
  const int sb = s / a.W, w = s % a.W;
  const int r0 = g.row0 + sb * RS1;
  const int rn = min(RS1, g.rcnt - sb * RS1);
  const unsigned rowbytes = (unsigned)g.nf4 * 16u;
  const unsigned qbytes = (unsigned)g.nf4 * 16u * RP;
  const unsigned pbytes = ((unsigned)(g.rcnt * RP * 4) + 15u) & ~15u;
  const bool prev = a.has_prev != 0;
  unsigned tx = 2u * (unsigned)rn * rowbytes + (prev ? qbytes : 0u);
  if (s == 0) tx += qbytes + (prev ? pbytes : 0u);
  if (lane == 0) mbar_expect_tx(wp.bar + slot, tx);
  __syncwarp();
  const int64_t col = (int64_t)4 * g.f0;
  char* hd = wp.hdr + hb * wp.hdr_bytes;
  if (lane < rn) {
    const float* src = a.G[w] + L.off + (int64_t)(r0 + lane) * L.ld + col;
    bulk_g2s(sl + lane * rowbytes, src, rowbytes, wp.bar + slot, wp.pol_first);
  } else if (lane >= 8 && lane - 8 < rn) {
    const float* src = a.B + (int64_t)w * a.total + L.off + (int64_t)(r0 + lane - 8) * L.ld + col;
    bulk_g2s(sl + RS1 * NF4 * 16 + (lane - 8) * rowbytes, src, rowbytes, wp.bar + slot, wp.pol_first);
  } else if (lane == 16 && prev) {
    const float* src = a.Qw + (int64_t)w * a.q_total + L.q_off + col * RP;
    bulk_g2s(sl + 2 * RS1 * NF4 * 16, src, qbytes, wp.bar + slot, wp.pol_first);
  } else if (lane == 17 && s == 0) {
    bulk_g2s(hd, a.Qbar + L.q_off + col * RP, qbytes, wp.bar + slot, wp.pol_first);
  } else if (lane == 18 && s == 0 && prev) {
    bulk_g2s(hd + Cfg<RP>::QSPAN, a.Phat + L.p_off + (int64_t)g.row0 * RP, pbytes, wp.bar + slot, wp.pol_first);
  }
  ++wp.head;
}

// One P1 item (row block rb, column span sg).  `claim` (lane 0) is the next
// item of this warp: when it is a P1 item too, its first stages are issued
// while this item drains, so the warp's copy stream never runs dry.
template <int RP>
__device__ bool p1_item(const StepArgs& a, const LayerDev& L, int it, int rb, int sg, unsigned claim,
                        WarpPipe& wp) {
  constexpr int RS1 = Cfg<RP>::RS1;
  constexpr int NF4 = Cfg<RP>::NF4;
  constexpr int NST = Cfg<RP>::NST;
  const int lane = threadIdx.x & 31;
  const P1Geo g = p1_geo<RP>(L, rb, sg);
  const int ns = g.nsb * a.W;
  const int hb = wp.hb;
  wp.hb ^= 1;
  int issued = (wp.pre_item == it) ? wp.pre_count : 0;
  wp.pre_item = -1;
  wp.pre_count = 0;
  while (issued < ns && wp.head - wp.tail < (unsigned)NST) p1_issue<RP>(a, L, g, issued++, hb, wp);

  // the next item, for prefetching
  const unsigned nx = __shfl_sync(kFull, claim, 0);
  bool nx_p1 = false;
  int nx_layer = 0, nx_ns = 0;
  P1Geo g2;
  if (nx < (unsigned)a.num_items) {
    const Item ni = a.items[nx];
    if (ni.kind == kItemP1) {
      nx_p1 = true;
      nx_layer = ni.layer;
      g2 = p1_geo<RP>(a.layers[ni.layer], ni.a, ni.b);
      nx_ns = g2.nsb * a.W;
    }
  }

  const float* hd = reinterpret_cast<const float*>(wp.hdr + hb * wp.hdr_bytes);  // Qbar span
  const float* pp = hd + Cfg<RP>::QSPAN / 4;                                    // previous Phat rows
  const bool prev = a.has_prev != 0;
  float acc[RS1][RP];
  for (int s = 0; s < ns; ++s) {
    int slot;
    if (!ring_pop<NST>(wp, a.ctl, a.spin_limit, it, slot)) return false;
    const int sb = s / a.W, w = s % a.W;
    if (w == 0) {
#pragma unroll
      for (int i = 0; i < RS1; ++i)
#pragma unroll
        for (int k = 0; k < RP; ++k) acc[i][k] = 0.f;
    }
    const int rl = sb * RS1;  // first row of the sub-block within the item
    const int rn = min(RS1, g.rcnt - rl);
    const char* sl = wp.ring + slot * wp.slot_bytes;
    const float4* sG = reinterpret_cast<const float4*>(sl);
    const float4* sB = reinterpret_cast<const float4*>(sl + RS1 * NF4 * 16);
    const float* sQw = reinterpret_cast<const float*>(sl + 2 * RS1 * NF4 * 16);
    float* Bw = a.B + (int64_t)w * a.total + L.off;
    for (int cc = lane; cc < g.nf4; cc += 32) {
      const int c = g.f0 + cc;  // float4 column in the row
      const bool tailc = (c == L.F - 1) && (L.tail < 4);
      float qw[4][RP], qv[4][RP];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < RP; ++k) {
          qw[j][k] = prev ? sQw[(cc * 4 + j) * RP + k] : 0.f;
          qv[j][k] = hd[(cc * 4 + j) * RP + k];
        }
#pragma unroll
      for (int i = 0; i < RS1; ++i) {
        if (i < rn) {
          const float4 gv = sG[i * g.nf4 + cc];
          const float4 bv = sB[i * g.nf4 + cc];
          // E_w = B_w - Phat' Q_w'^T, k ascending (the same chain as the
          // error read-back kernel)
          float e0 = bv.x, e1 = bv.y, e2 = bv.z, e3 = bv.w;
          if (prev) {
#pragma unroll
            for (int k = 0; k < RP; ++k) {
              const float p = pp[(rl + i) * RP + k];
              e0 = fmaf(-p, qw[0][k], e0);
              e1 = fmaf(-p, qw[1][k], e1);
              e2 = fmaf(-p, qw[2][k], e2);
              e3 = fmaf(-p, qw[3][k], e3);
            }
          }
          float m0 = gv.x + e0, m1 = gv.y + e1, m2 = gv.z + e2, m3 = gv.w + e3;
          if (tailc) {
            if (L.tail < 2) m1 = 0.f;
            if (L.tail < 3) m2 = 0.f;
            m3 = 0.f;
          }
          *reinterpret_cast<float4*>(Bw + (int64_t)(g.row0 + rl + i) * L.ld + 4 * c) = make_float4(m0, m1, m2, m3);
#pragma unroll
          for (int k = 0; k < RP; ++k) {
            float t = acc[i][k];
            t = fmaf(m0, qv[0][k], t);
            t = fmaf(m1, qv[1][k], t);
            t = fmaf(m2, qv[2][k], t);
            t = fmaf(m3, qv[3][k], t);
            acc[i][k] = t;
          }
        }
      }
    }
    __syncwarp();
    ++wp.tail;
    // refill the freed slot: this item's next stage, else the next item's
    if (issued < ns) {
      fence_proxy_async_smem();
      p1_issue<RP>(a, L, g, issued++, hb, wp);
    } else if (nx_p1 && wp.pre_count < nx_ns) {
      fence_proxy_async_smem();
      p1_issue<RP>(a, a.layers[nx_layer], g2, wp.pre_count, wp.hb, wp);
      wp.pre_item = (int)nx;
      ++wp.pre_count;
    }
    if (w == a.W - 1) {
      // the sub-block is complete: reduce over the lanes (fixed butterfly)
#pragma unroll
      for (int i = 0; i < RS1; ++i)
#pragma unroll
        for (int k = 0; k < RP; ++k) {
          const float v = warp_sum(acc[i][k]);
          if (lane == 0 && i < rn) wp.prow[(rl + i) * RP + k] = v;
        }
    }
  }
  __syncwarp();
  float* s_prow = wp.prow;
  if (L.nsg1 > 1) {
    float* pp2 = a.ppart + L.ppart_off + ((int64_t)rb * L.nsg1 + sg) * Cfg<RP>::R1 * RP;
    for (int idx = lane; idx < g.rcnt * RP; idx += 32) pp2[idx] = s_prow[idx];
    if (!warp_arrive_last(a.counters + L.cnt_off + L.c_rb + rb, (unsigned)L.nsg1)) return true;
    const float* pb = a.ppart + L.ppart_off + (int64_t)rb * L.nsg1 * Cfg<RP>::R1 * RP;
    for (int idx = lane; idx < g.rcnt * RP; idx += 32) {
      float t = 0.f;
      for (int q = 0; q < L.nsg1; ++q) t += __ldcg(pb + (int64_t)q * Cfg<RP>::R1 * RP + idx);
      s_prow[idx] = t;
    }
    __syncwarp();
  }
  for (int idx = lane; idx < g.rcnt * RP; idx += 32) a.P[L.p_off + (int64_t)g.row0 * RP + idx] = s_prow[idx];
  __syncwarp();
  gram_tail<RP>(a, L, rb, s_prow, g.rcnt);
  return true;
}

// ----------------------------------------------------------------------------
// PH: Phat rows by forward substitution Phat R = P (float64)
// ----------------------------------------------------------------------------
template <int RP>
__device__ void ph_item(const StepArgs& a, const LayerDev& L, int item) {
  const int lane = threadIdx.x & 31;
  const int row = item * 32 + lane;
  const double* R = a.rinv + L.rinv_off;
  if (row < L.n) {
    double x[RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) x[k] = (double)__ldcg(a.P + L.p_off + (int64_t)row * RP + k);
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      double s = x[k];
#pragma unroll
      for (int j = 0; j < k; ++j) s = fma(-x[j], __ldcg(R + j * RP + k), s);
      x[k] = s * __ldcg(R + RP * RP + k);
    }
    float* out = a.Phat + L.p_off + (int64_t)row * RP;
#pragma unroll
    for (int k = 0; k < RP; ++k) out[k] = (float)x[k];
  }
  if (warp_arrive_last(a.counters + L.cnt_off + L.c_ph, (unsigned)L.tph))
    warp_publish(&a.flags[L.flag_off + 1], a.epoch);
}

// ----------------------------------------------------------------------------
// P3: partial Q_w = M_w^T Phat over r3 rows of one segment; segment finalise
// ----------------------------------------------------------------------------
// The last row tile of (segment, worker) sums the partial Q_w of the
// segment's columns over the row tiles (fixed order); the last worker of the
// segment then forms Qbar = mean_w Q_w; the last segment publishes Qbar.
template <int RP>
__device__ void qf_segment_worker(const StepArgs& a, const LayerDev& L, int seg, int w) {
  const int lane = threadIdx.x & 31;
  const int col0 = seg * kSeg * 4;
  const int col1 = min(L.ld, col0 + kSeg * 4);
  const int n4 = (col1 - col0) * RP / 4;  // float4 of the segment's ld x RP slice
  const int64_t e0 = (int64_t)col0 * RP;
  const int64_t wstride = (int64_t)L.ld * RP;
  const float* parts = a.qpart + L.qpart_off + (int64_t)w * wstride + e0;
  float* qw = a.Qw + (int64_t)w * a.q_total + L.q_off + e0;
  const int64_t tstride = (int64_t)a.W * wstride;  // from one row tile to the next
  for (int q = lane; q < n4; q += 32) {
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
  if (!warp_arrive_last(a.counters + L.cnt_off + L.c_qs + seg, (unsigned)a.W)) return;
  const float invw = 1.0f / (float)a.W;
  for (int q = lane; q < n4; q += 32) {
    float4 s = zero4();
    for (int v = 0; v < a.W; ++v) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(a.Qw + (int64_t)v * a.q_total + L.q_off + e0) + q);
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    reinterpret_cast<float4*>(a.Qbar + L.q_off + e0)[q] =
        make_float4(s.x * invw, s.y * invw, s.z * invw, s.w * invw);
  }
  if (warp_arrive_last(a.counters + L.cnt_off + L.c_qf, (unsigned)L.S))
    warp_publish(&a.flags[L.flag_off + 2], a.epoch);
}

template <int RP>
__device__ bool p3_item(const StepArgs& a, const LayerDev& L, int it, int rt, int segw, WarpPipe& wp) {
  constexpr int R3C = Cfg<RP>::R3C;
  constexpr int NST = Cfg<RP>::NST;
  const int lane = threadIdx.x & 31;
  const int seg = segw / a.W, w = segw % a.W;
  const int row0 = rt * L.r3;
  const int nrows = min(L.r3, L.n - row0);
  const int nf4 = min(kSeg, L.F - seg * kSeg);
  const unsigned rowbytes = (unsigned)nf4 * 16u;
  const int nch = (nrows + R3C - 1) / R3C;
  const float* Bw = a.B + (int64_t)w * a.total + L.off + 4 * seg * kSeg;
  const float* Ph = a.Phat + L.p_off;
  // chunk t: lanes [0, rn) copy their B row, lane 16 the Phat rows
  auto issue = [&](int t) {
    const int slot = (int)(wp.head % NST);
    char* sl = wp.ring + slot * wp.slot_bytes;
    const int r = t * R3C;
    const int rn = min(R3C, nrows - r);
    const unsigned pbytes = ((unsigned)(rn * RP * 4) + 15u) & ~15u;
    if (lane == 0) mbar_expect_tx(wp.bar + slot, (unsigned)rn * rowbytes + pbytes);
    __syncwarp();
    if (lane < rn)
      bulk_g2s(sl + lane * kSeg * 16, Bw + (int64_t)(row0 + r + lane) * L.ld, rowbytes, wp.bar + slot, wp.pol_first);
    else if (lane == 16)
      bulk_g2s(sl + R3C * kSeg * 16, Ph + (int64_t)(row0 + r) * RP, pbytes, wp.bar + slot, wp.pol_first);
    ++wp.head;
  };
  // B and Phat were written by other warps of this launch (generic proxy)
  fence_proxy_async_global();
  int issued = 0;
  while (issued < nch && wp.head - wp.tail < (unsigned)NST) issue(issued++);

  float acc[4][RP];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < RP; ++k) acc[j][k] = 0.f;
  const bool act = lane < nf4;
  for (int t = 0; t < nch; ++t) {
    int slot;
    if (!ring_pop<NST>(wp, a.ctl, a.spin_limit, it, slot)) return false;
    const int rn = min(R3C, nrows - t * R3C);
    const char* sl = wp.ring + slot * wp.slot_bytes;
    const float4* sb = reinterpret_cast<const float4*>(sl);
    const float* sp = reinterpret_cast<const float*>(sl + R3C * kSeg * 16);
    if (act) {
#pragma unroll
      for (int u = 0; u < R3C; ++u) {
        if (u < rn) {
          const float4 b = sb[u * kSeg + lane];
#pragma unroll
          for (int k = 0; k < RP; ++k) {
            const float p = sp[u * RP + k];
            acc[0][k] = fmaf(b.x, p, acc[0][k]);
            acc[1][k] = fmaf(b.y, p, acc[1][k]);
            acc[2][k] = fmaf(b.z, p, acc[2][k]);
            acc[3][k] = fmaf(b.w, p, acc[3][k]);
          }
        }
      }
    }
    __syncwarp();
    ++wp.tail;
    if (issued < nch) {
      fence_proxy_async_smem();
      issue(issued++);
    }
  }
  if (act) {
    const int c = seg * kSeg + lane;
    float* part = a.qpart + L.qpart_off + ((int64_t)rt * a.W + w) * L.ld * RP + (int64_t)(4 * c) * RP;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if constexpr (RP % 4 == 0) {
#pragma unroll
        for (int k = 0; k < RP; k += 4)
          *reinterpret_cast<float4*>(part + j * RP + k) =
              make_float4(acc[j][k], acc[j][k + 1], acc[j][k + 2], acc[j][k + 3]);
      } else {
#pragma unroll
        for (int k = 0; k < RP; ++k) part[j * RP + k] = acc[j][k];
      }
    }
  }
  if (warp_arrive_last(a.counters + L.cnt_off + L.c_p3 + seg * a.W + w, (unsigned)L.t3r))
    qf_segment_worker<RP>(a, L, seg, w);
  return true;
}

// ----------------------------------------------------------------------------
// U: rows of Phat Qbar^T
// ----------------------------------------------------------------------------
template <int RP>
__device__ bool u_item(const StepArgs& a, const LayerDev& L, int it, int rb, int sg, WarpPipe& wp) {
  constexpr int RS = Cfg<RP>::RSU;
  constexpr int GSU = Cfg<RP>::GSU;
  constexpr int NST = Cfg<RP>::NST;
  const int lane = threadIdx.x & 31;
  const int row0 = rb * RS;
  const int rcnt = min(RS, L.n - row0);
  const int f0 = sg * GSU * kSeg;
  const int nf4 = min(GSU * kSeg, L.F - f0);
  float* s_ph = wp.prow;  // RS x RP
  const unsigned qbytes = (unsigned)nf4 * 16u * RP;
  fence_proxy_async_global();  // Qbar was written by other warps of this launch
  const int islot = (int)(wp.head % NST);
  float* s_q = reinterpret_cast<float*>(wp.ring + islot * wp.slot_bytes);  // Qbar rows 4 f0 .. 4 (f0 + nf4)
  if (lane == 0) {
    mbar_expect_tx(wp.bar + islot, qbytes);
    bulk_g2s(s_q, a.Qbar + L.q_off + (int64_t)4 * f0 * RP, qbytes, wp.bar + islot, wp.pol_first);
  }
  ++wp.head;
  for (int i = lane; i < rcnt * RP; i += 32) s_ph[i] = __ldcg(a.Phat + L.p_off + (int64_t)row0 * RP + i);
  int slot;
  if (!ring_pop<NST>(wp, a.ctl, a.spin_limit, it, slot)) return false;
  __syncwarp();
  for (int cc = lane; cc < nf4; cc += 32) {
    float qv[4][RP];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < RP; ++k) qv[j][k] = s_q[(cc * 4 + j) * RP + k];
    float* Ub = a.U + L.off + 4 * (f0 + cc);
#pragma unroll
    for (int i = 0; i < RS; ++i) {
      if (i < rcnt) {
        float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
        for (int k = 0; k < RP; ++k) {
          const float p = s_ph[i * RP + k];
          u0 = fmaf(p, qv[0][k], u0);
          u1 = fmaf(p, qv[1][k], u1);
          u2 = fmaf(p, qv[2][k], u2);
          u3 = fmaf(p, qv[3][k], u3);
        }
        __stcs(reinterpret_cast<float4*>(Ub + (int64_t)(row0 + i) * L.ld), make_float4(u0, u1, u2, u3));
      }
    }
  }
  __syncwarp();
  ++wp.tail;
  return true;
}

// ----------------------------------------------------------------------------
// V: worker mean of a vector layer
// ----------------------------------------------------------------------------
__device__ __forceinline__ void v_item(const StepArgs& a, const VecDev& V, int item) {
  const int base = item * kVChunk;
  const int end = min(V.n, base + kVChunk);
  for (int i = base + (int)(threadIdx.x & 31); i < end; i += 32) {
    float s = 0.f;
    for (int w = 0; w < a.W; ++w) s += __ldcs(a.G[w] + V.off + i);
    a.U[V.off + i] = s / (float)a.W;
  }
}

// ----------------------------------------------------------------------------
// the persistent step kernel: every warp drains the queue on its own
// ----------------------------------------------------------------------------
template <int RP>
__global__ void __launch_bounds__(kThreads, Cfg<RP>::MINB) step_kernel(const StepArgs a) {
  extern __shared__ __align__(128) char smem[];
  constexpr int NST = Cfg<RP>::NST;
  const int lane = threadIdx.x & 31;
  WarpPipe wp;
  char* mine = smem + (threadIdx.x >> 5) * Cfg<RP>::WSM_BYTES;
  wp.bar = reinterpret_cast<uint64_t*>(mine);
  wp.ring = mine + Cfg<RP>::BAR_BYTES;
  wp.slot_bytes = Cfg<RP>::SLOT;
  wp.hdr_bytes = ((Cfg<RP>::HDR + 15) / 16) * 16;
  wp.hdr = wp.ring + NST * Cfg<RP>::SLOT;
  wp.prow = reinterpret_cast<float*>(wp.hdr + 2 * wp.hdr_bytes);
  wp.phase = 0u;
  wp.head = wp.tail = 0u;
  wp.pre_item = -1;
  wp.pre_count = 0;
  wp.hb = 0;
  wp.pol_first = policy_evict_first();
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NST; ++i) mbar_init(wp.bar + i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  unsigned claim = 0;
  if (lane == 0) claim = atomicAdd(&a.ctl->next, 1u);
  claim = __shfl_sync(kFull, claim, 0);
  for (;;) {
    const unsigned it = claim;
    if (it >= (unsigned)a.num_items) break;
    // claim the next item now; its index is only read after this one is done
    if (lane == 0) claim = atomicAdd(&a.ctl->next, 1u);
    const Item item = a.items[it];
    bool ok = true;
    uint64_t t0 = 0, tw = 0;
    if (a.trace != nullptr) t0 = tw = globaltimer_ns();
    if (item.kind == kItemV) {
      if (a.U != nullptr) v_item(a, a.vecs[item.layer], item.a);
    } else {
      const LayerDev& L = a.layers[item.layer];
      switch (item.kind) {
        case kItemP1:
          ok = p1_item<RP>(a, L, (int)it, item.a, item.b, claim, wp);
          break;
        case kItemPH:
          if (warp_wait(&a.flags[L.flag_off + 0], a.epoch, a.ctl, a.spin_limit, (int)it)) {
            if (a.trace != nullptr) tw = globaltimer_ns();
            ph_item<RP>(a, L, item.a);
          }
          break;
        case kItemP3:
          if (warp_wait(&a.flags[L.flag_off + 1], a.epoch, a.ctl, a.spin_limit, (int)it)) {
            if (a.trace != nullptr) tw = globaltimer_ns();
            ok = p3_item<RP>(a, L, (int)it, item.a, item.b, wp);
          }
          break;
        case kItemU:
          if (a.U != nullptr && warp_wait(&a.flags[L.flag_off + 2], a.epoch, a.ctl, a.spin_limit, (int)it)) {
            if (a.trace != nullptr) tw = globaltimer_ns();
            ok = u_item<RP>(a, L, (int)it, item.a, item.b, wp);
          }
          break;
        default:
          break;
      }
    }
    if (a.trace != nullptr && lane == 0) {
      TraceRec r;
      r.item = it;
      r.sm = (uint16_t)smid();
      r.warp = (uint16_t)((blockIdx.x * kWarps + (threadIdx.x >> 5)) & 0xffff);
      r.t0 = t0;
      r.tw = tw;
      r.t1 = globaltimer_ns();
      a.trace[it] = r;
    }
    claim = __shfl_sync(kFull, claim, 0);
    if (!ok) break;  // a bulk copy never landed: the error is recorded, stop
  }
  // copies issued ahead for an item this warp will not run: let them land
  // (bounded) before the warp's shared memory is released
  while (wp.head != wp.tail) {
    int slot;
    if (!ring_pop<NST>(wp, a.ctl, a.spin_limit, -1, slot)) break;
    ++wp.tail;
  }
  if (lane == 0) {
    __threadfence();
    const unsigned e = atomicAdd(&a.ctl->exited, 1u);
    if (e == gridDim.x * kWarps - 1) {
      a.ctl->next = 0u;
      a.ctl->exited = 0u;
    }
  }
}

// Dynamic shared memory of the step kernel.
template <int RP>
size_t step_smem_bytes() {
  return (size_t)kWarps * Cfg<RP>::WSM_BYTES;
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
  if (threadIdx.x < 32) warp_wait(flag, 1u, ctl, limit, 0);
}
#endif  // PSGD_SIDE_KERNELS

}  // namespace psgd
