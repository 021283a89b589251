// libspecverify: the speculative-decoding verification sampler for GB300
// (sm_103a).  One persistent kernel does the whole step.
//
// The rule ("Decodificación Especulativa y EAGLE", Phase 10 - Lesson 25,
// sections "El Concepto", "La Regla de Exactitud", "Caso codicioso"): for
// each request, accept drafted tokens left to right while u_t < p(x_t)/q(x_t);
// at the first rejection draw a replacement from (p - q)+ and stop; if every
// draft is accepted draw a bonus token from p at the next position; at
// temperature 0 compare argmax(p) with the draft instead.
//
// Work unit = one (request b, position t): target row t, plus draft row t
// when t < n_b and T_b > 0.  A thread-block cluster of C CTAs handles one
// unit at a time, CTA c owning vocabulary slice c; the grid holds as many
// clusters as fit on the GPU and each loops over units taken from a ticket
// counter.  Inside a CTA:
//   * a producer warp prefetches the slices of upcoming units into a ring of
//     shared-memory stages with TMA bulk copies (full / empty mbarriers);
//     cluster rank 0 takes the tickets and sends each unit's description to
//     every producer of its cluster with st.async;
//   * eight consumer warps make one pass over a stage: the slice maximum and
//     the sum of exp((z - max)/T) (online), or the argmax at T = 0; the CTA's
//     partial goes to every CTA of the cluster with st.async, so each CTA
//     combines all partials in the same order and takes the same decisions;
//   * if the position can be the request's final draw (a rejection, or the
//     bonus position) the consumers draw by inverse CDF over the residual
//     (p - q)+ or over p, from the slices still in shared memory;
//   * the CTA that produced the unit's result stores a record and bumps the
//     request's counter (acq_rel); the last unit of a request to arrive
//     writes accepted_len and out_tokens.  Nobody waits for another unit.
// Every logit the rule needs is read from HBM once.  Every wait on an
// mbarrier is bounded in time; a timeout sets a status bit and the kernel
// drains and exits.

#include <cooperative_groups.h>
#include <cuda/atomic>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "specverify.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;               // + one producer warp
constexpr int kMaxCluster = 16;
constexpr int kMaxStages = 6;
constexpr int kChunkBytes = 16;                         // one 128-bit vector
constexpr int kSliceMaxBytes = 96 * 1024;               // per row per CTA
constexpr int kMaxChunks = kSliceMaxBytes / kChunkBytes + 1;
constexpr int kMaxTiles = (kMaxChunks + kConsumers - 1) / kConsumers;
constexpr long long kWaitLimitCycles = 4000000000ll;   // ~2 s per wait at 2 GHz
constexpr uint32_t kSuspendHintNs = 1000000;           // 1 ms sleep per try

constexpr int kRecAccept = 1;
constexpr int kRecBad = 2;

constexpr int kWsStatus = 0;   // workspace header (int32 words)
constexpr int kWsWork = 1;     // next unit ticket
constexpr int kWsExit = 2;     // CTAs that finished

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  const float* uniforms;
  const float* uniforms_resample;
  int B, K, V;
  int units;               // B * (K + 1)
  int slice;               // vocabulary elements per CTA (multiple of the chunk)
  int slice_bytes;         // shared-memory bytes per row slice (16 B phase room)
  int stage_bytes;         // one stage: target slice (+ draft slice)
  int stages;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t* header;         // status, ticket, exit count
  int32_t* counters;       // [B]
  int2* records;           // [B, K+1]
  float* row_stats;        // [B, K+1, 8] or null
};

// One unit as the producer of cluster rank 0 hands it out (32 bytes).
struct __align__(16) Meta {
  int u, b, t, n;
  float T, u_t, u_draw;
  int x;
};

// One CTA's partial result for a unit (32 bytes).
//   sampled: a = {max_p, sum_p, max_q, sum_q}, b = {z_p[x], z_q[x], -, -}
//   greedy:  a = {best value, best index (bits), -, -}
struct __align__(16) Part {
  float4 a, b;
};

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t meta_bar[kMaxStages];
  uint64_t x1_bar[2];
  uint64_t x2_bar[2][2];
  Meta inbox[kMaxStages];   // written by rank 0's producer (st.async)
  Meta cmeta[kMaxStages];   // the unit in each stage, for the consumers
  Part x1[2][kMaxCluster];
  float x2[2][2][kMaxCluster];
  float4 red[kConsumerWarps];
  float ws[kMaxTiles * kConsumerWarps];
  int pabort;   // written by the producer warp only
  int cabort;   // written by consumer threads only (read after a consumer barrier)
  int sel_tile, sel_warp;
  float tau_warp;
};

// ---------------------------------------------------------------- elements

template <int DT> struct Elt;
template <> struct Elt<SPECV_F32> {
  static constexpr int kBytes = 4;
  static constexpr int kPerChunk = 4;
  __device__ static void unpack(uint4 raw, float v[4]) {
    v[0] = __uint_as_float(raw.x);
    v[1] = __uint_as_float(raw.y);
    v[2] = __uint_as_float(raw.z);
    v[3] = __uint_as_float(raw.w);
  }
  __device__ static float chunk_max(uint4 raw) {
    return fmaxf(fmaxf(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                 fmaxf(__uint_as_float(raw.z), __uint_as_float(raw.w)));
  }
  __device__ static void copy1(unsigned char* dst, const unsigned char* src) {
    *reinterpret_cast<float*>(dst) = __ldg(reinterpret_cast<const float*>(src));
  }
};
template <> struct Elt<SPECV_BF16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerChunk = 8;
  __device__ static void unpack(uint4 raw, float v[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  // Maximum of the 8 bf16 values with packed bf16x2 max, then widened.
  __device__ static float chunk_max(uint4 raw) {
    uint32_t m01, m23, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m01) : "r"(raw.x), "r"(raw.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m23) : "r"(raw.z), "r"(raw.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m01), "r"(m23));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ static void copy1(unsigned char* dst, const unsigned char* src) {
    *reinterpret_cast<unsigned short*>(dst) = __ldg(reinterpret_cast<const unsigned short*>(src));
  }
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t peer_addr(const void* p, int rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(p)), "r"(rank));
  return out;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Tests phase `parity`; a thread whose phase is not complete sleeps in the
// instruction until it completes or about kSuspendHintNs pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of the barrier; gives up after kWaitLimitCycles
// SM clock cycles (about two seconds).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// Non-tensor TMA bulk copy global -> this CTA's shared memory.  Both
// addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  const unsigned long long gsrc = static_cast<unsigned long long>(__cvta_generic_to_global(src));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte store into another CTA's shared memory, completing tx on its mbarrier.
__device__ __forceinline__ void st_async16(uint32_t remote, uint32_t remote_bar, uint32_t a,
                                           uint32_t b, uint32_t c, uint32_t d) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(remote),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(remote_bar)
      : "memory");
}

__device__ __forceinline__ void st_async4(uint32_t remote, uint32_t remote_bar, uint32_t a) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   remote),
               "r"(a), "r"(remote_bar)
               : "memory");
}

// Barrier among the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// 2^x on the MUFU unit (PTX ex2.approx.ftz.f32); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp((z - m)/T) as 2^((z - m) * log2(e)/T), the argument formed exactly
// from the difference to the reference m.
__device__ __forceinline__ float scaled_exp(float z, float m, float sT) {
  return ex2(__fmul_rn(__fsub_rn(z, m), sT));
}

// ---------------------------------------------------------------- reductions

// Online (max, sum of exp) pairs: the sum is relative to the max.
__device__ __forceinline__ void pair_combine(float& m, float& s, float om, float os, float sT) {
  const float M = fmaxf(m, om);
  if (M == -INFINITY) { m = M; s = 0.0f; return; }
  s = __fadd_rn(__fmul_rn(s, scaled_exp(m, M, sT)), __fmul_rn(os, scaled_exp(om, M, sT)));
  m = M;
}

__device__ __forceinline__ void warp_pair(float& m, float& s, float sT) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    pair_combine(m, s, om, os, sT);
  }
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = __fadd_rn(v, y);
  }
  return v;
}

// ---------------------------------------------------------------- slices

// Where a unit's row slice sits: the slice holds elements [e0, e0 + cnt) of
// the row; shared memory keeps the global 16-byte phase h, so element i of
// the slice is at byte h + i * elt and chunk j covers bytes [16 j, 16 j + 16).
struct SliceGeo {
  int e0, cnt, h, nch;
};

template <int DT>
__device__ __forceinline__ SliceGeo slice_geo(const Params& P, const void* base, size_t row,
                                              int crank) {
  using E = Elt<DT>;
  SliceGeo g;
  g.e0 = crank * P.slice;
  g.cnt = max(0, min(P.slice, P.V - g.e0));
  const uintptr_t gsrc = reinterpret_cast<uintptr_t>(base) +
                         (row * static_cast<size_t>(P.V) + g.e0) * E::kBytes;
  g.h = static_cast<int>(gsrc & 15);
  g.nch = (g.h + g.cnt * E::kBytes + 15) / 16;
  return g;
}

// Slice-local index of the first element of chunk j (may be negative).
template <int DT>
__device__ __forceinline__ int chunk_base(const SliceGeo& g, int j) {
  return (16 * j - g.h) / Elt<DT>::kBytes;
}

template <int DT>
__device__ __forceinline__ bool chunk_full(const SliceGeo& g, int j) {
  const int i0 = chunk_base<DT>(g, j);
  return i0 >= 0 && i0 + Elt<DT>::kPerChunk <= g.cnt;
}

// ---------------------------------------------------------------- producer

__device__ __forceinline__ Meta sentinel_meta() {
  Meta m;
  m.u = -1;
  m.b = m.t = m.n = m.x = 0;
  m.T = m.u_t = m.u_draw = 0.0f;
  return m;
}

// Warp-collective: resolve tickets until one names a unit with work.
// Requests with bad data are answered here (by their position-0 ticket).
__device__ Meta resolve_ticket(const Params& P, int ticket, int lane) {
  const int B = P.B, K = P.K, V = P.V;
  for (;;) {
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    if (ticket >= P.units) return sentinel_meta();
    const int t = ticket / B;
    const int b = ticket - t * B;
    const int n = P.draft_len ? __ldg(P.draft_len + b) : K;
    const float T = __ldg(P.temperature + b);
    int bad = 0;
    if (n < 1 || n > K) {
      bad = SPECV_DEV_BAD_DRAFT_LEN;
    } else {
      if (!(T >= 0.0f) || isinf(T)) bad |= SPECV_DEV_BAD_TEMPERATURE;
      if (T > 0.0f && P.draft == nullptr) bad |= SPECV_DEV_NO_DRAFT;
      int tok_bad = 0, u_bad = 0;
      if (lane < n) {
        const int x = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + lane);
        tok_bad = (x < 0 || x >= V);
      }
      if (lane <= n) {
        const float u = __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + lane);
        u_bad = !(u >= 0.0f && u < 1.0f);
      }
      if (__any_sync(0xffffffffu, tok_bad)) bad |= SPECV_DEV_BAD_TOKEN;
      const float ur = __ldg(P.uniforms_resample + b);
      if (__any_sync(0xffffffffu, u_bad) || !(ur >= 0.0f && ur < 1.0f)) bad |= SPECV_DEV_BAD_UNIFORM;
    }
    if (bad || t > n) {
      if (bad && t == 0 && lane == 0) {
        atomicOr(P.header + kWsStatus, bad);
        P.accepted_len[b] = -1;
        for (int s = 0; s <= K; ++s) P.out_tokens[static_cast<size_t>(b) * (K + 1) + s] = -1;
      }
      if (lane == 0) ticket = atomicAdd(P.header + kWsWork, 1);
      continue;
    }
    Meta m;
    m.u = ticket;
    m.b = b;
    m.t = t;
    m.n = n;
    m.T = T;
    m.x = t < n ? __ldg(P.draft_tokens + static_cast<size_t>(b) * K + t) : -1;
    m.u_t = t < n ? __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + t) : 0.0f;
    m.u_draw = t < n ? __ldg(P.uniforms_resample + b)
                     : __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + n);
    return m;
  }
}

// Copies one row slice into shared memory: the 16-byte-aligned interior by
// one bulk copy (issued later by lane 0), the unaligned head and tail by
// the lanes.  Returns the bulk byte count; *bulk_src / *bulk_dst describe it.
template <int DT>
__device__ uint32_t stage_row(const Params& P, const void* base, size_t row, int crank,
                              unsigned char* dst, int lane, const unsigned char** bulk_src,
                              unsigned char** bulk_dst) {
  using E = Elt<DT>;
  const SliceGeo g = slice_geo<DT>(P, base, row, crank);
  const unsigned char* gsrc = static_cast<const unsigned char*>(base) +
                              (row * static_cast<size_t>(P.V) + g.e0) * E::kBytes;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(gsrc);
  const uintptr_t s1 = s0 + static_cast<uintptr_t>(g.cnt) * E::kBytes;
  const uintptr_t a = (s0 + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t z = s1 & ~static_cast<uintptr_t>(15);
  uint32_t bulk = 0;
  uintptr_t head_end = s1, tail_begin = s1;
  if (a < z) {
    bulk = static_cast<uint32_t>(z - a);
    *bulk_src = reinterpret_cast<const unsigned char*>(a);
    *bulk_dst = dst + g.h + (a - s0);
    head_end = a;
    tail_begin = z;
  }
  // head [s0, head_end) and tail [tail_begin, s1): element copies
  const int nhead = static_cast<int>((head_end - s0) / E::kBytes);
  const int ntail = static_cast<int>((s1 - tail_begin) / E::kBytes);
  for (int i = lane; i < nhead + ntail; i += 32) {
    const uintptr_t off = i < nhead ? static_cast<uintptr_t>(i) * E::kBytes
                                    : (tail_begin - s0) + static_cast<uintptr_t>(i - nhead) * E::kBytes;
    E::copy1(dst + g.h + off, gsrc + off);
  }
  return bulk;
}

template <int DT>
__device__ void producer(const Params& P, Ctl& S, unsigned char* dyn, int crank, int C, int lane) {
  Meta next = sentinel_meta();
  if (crank == 0) {
    int ticket = 0;
    if (lane == 0) ticket = atomicAdd(P.header + kWsWork, 1);
    next = resolve_ticket(P, ticket, lane);
  }
  for (int k = 0;; ++k) {
    const int s = k % P.stages;
    const uint32_t ph = static_cast<uint32_t>(k / P.stages) & 1u;
    int ticket = 0;
    bool ok = true;
    if (crank == 0) {
      // Stage s is free here once this CTA's consumers finished unit k - stages;
      // their exchange with every peer for that unit proves each peer's
      // producer has taken its inbox[s] too, so the inbox can be refilled.
      ok = __all_sync(0xffffffffu, mbar_wait(&S.empty[s], ph ^ 1u));
      const Meta m = ok ? next : sentinel_meta();
      if (m.u >= 0 && lane == 0) ticket = atomicAdd(P.header + kWsWork, 1);   // the following unit
      if (lane > 0 && lane < C) {
        const uint32_t dst = peer_addr(&S.inbox[s], lane);
        const uint32_t bar = peer_addr(&S.meta_bar[s], lane);
        st_async16(dst, bar, static_cast<uint32_t>(m.u), static_cast<uint32_t>(m.b),
                   static_cast<uint32_t>(m.t), static_cast<uint32_t>(m.n));
        st_async16(dst + 16, bar, __float_as_uint(m.T), __float_as_uint(m.u_t),
                   __float_as_uint(m.u_draw), static_cast<uint32_t>(m.x));
      }
      if (lane == 0) S.inbox[s] = m;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.meta_bar[s]);
    } else if (lane == 0) {
      mbar_arrive_expect_tx(&S.meta_bar[s], sizeof(Meta));
    }
    ok = __all_sync(0xffffffffu, mbar_wait(&S.meta_bar[s], ph)) && ok;
    Meta m = S.inbox[s];
    if (crank != 0) ok = __all_sync(0xffffffffu, mbar_wait(&S.empty[s], ph ^ 1u)) && ok;
    int stop = 0;
    if (lane == 0) stop = S.cabort;   // the consumers gave up: stop feeding them
    stop = __shfl_sync(0xffffffffu, stop, 0);
    if (!ok || stop) {
      if (lane == 0 && !ok) {
        S.pabort = 1;
        atomicOr(P.header + kWsStatus, SPECV_DEV_TIMEOUT);
      }
      m = sentinel_meta();
    }
    if (lane == 0) S.cmeta[s] = m;
    if (m.u < 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.full[s]);
      return;
    }
    unsigned char* stage = dyn + static_cast<size_t>(s) * P.stage_bytes;
    const bool has_q = m.T > 0.0f && m.t < m.n;
    const size_t trow = static_cast<size_t>(m.b) * (P.K + 1) + m.t;
    const size_t drow = static_cast<size_t>(m.b) * P.K + m.t;
    const unsigned char *src_p = nullptr, *src_q = nullptr;
    unsigned char *dst_p = nullptr, *dst_q = nullptr;
    const uint32_t bp = stage_row<DT>(P, P.target, trow, crank, stage, lane, &src_p, &dst_p);
    const uint32_t bq = has_q ? stage_row<DT>(P, P.draft, drow, crank, stage + P.slice_bytes, lane,
                                              &src_q, &dst_q)
                              : 0u;
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(&S.full[s], bp + bq);
      if (bp) bulk_copy_g2s(dst_p, src_p, bp, &S.full[s]);
      if (bq) bulk_copy_g2s(dst_q, src_q, bq, &S.full[s]);
    }
    if (crank == 0) next = resolve_ticket(P, ticket, lane);
  }
}

// ---------------------------------------------------------------- combine

// Stores a unit's record; the last unit of request b to arrive writes the
// request's outputs.  One thread per unit.
__device__ void finish_unit(const Params& P, const Meta& m, int cand, int flags) {
  const int K = P.K, b = m.b, n = m.n;
  P.records[static_cast<size_t>(b) * (K + 1) + m.t] = make_int2(cand, flags);
  cuda::atomic_ref<int, cuda::thread_scope_device> counter(P.counters[b]);
  const int prev = counter.fetch_add(1, cuda::memory_order_acq_rel);
  if (prev != n) return;
  const int2* rec = P.records + static_cast<size_t>(b) * (K + 1);
  int j = n;
  bool bad = false;
  for (int s = 0; s <= n; ++s) {
    const int2 r = __ldcg(rec + s);
    if (r.y & kRecBad) bad = true;
    if (s < n && j == n && !(r.y & kRecAccept)) j = s;
  }
  int32_t* out = P.out_tokens + static_cast<size_t>(b) * (K + 1);
  if (bad) {
    atomicOr(P.header + kWsStatus, SPECV_DEV_BAD_ROW);
    P.accepted_len[b] = -1;
    for (int s = 0; s <= K; ++s) out[s] = -1;
  } else {
    const int final_tok = __ldcg(rec + j).x;
    for (int s = 0; s < j; ++s) out[s] = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + s);
    out[j] = final_tok;
    for (int s = j + 1; s <= K; ++s) out[s] = -1;
    P.accepted_len[b] = j;
  }
  counter.store(0, cuda::memory_order_relaxed);   // ready for the next call
}

// ---------------------------------------------------------------- consumers

// Warp 0 keeps its partial locally and sends it to every other CTA of the
// cluster (lane c addresses rank c).
__device__ __forceinline__ void send_part(Ctl& S, int xp, int crank, int C, int lane,
                                          const Part& part) {
  if (lane == 0) S.x1[xp][crank] = part;
  if (lane < C && lane != crank) {
    const uint32_t dst = peer_addr(&S.x1[xp][crank], lane);
    const uint32_t bar = peer_addr(&S.x1_bar[xp], lane);
    st_async16(dst, bar, __float_as_uint(part.a.x), __float_as_uint(part.a.y),
               __float_as_uint(part.a.z), __float_as_uint(part.a.w));
    st_async16(dst + 16, bar, __float_as_uint(part.b.x), __float_as_uint(part.b.y),
               __float_as_uint(part.b.z), __float_as_uint(part.b.w));
  }
}

// Bounded wait by every consumer thread, then a consumer barrier; returns
// false (for every consumer alike) if any of them gave up.
__device__ __forceinline__ bool consumers_wait(Ctl& S, const Params& P, uint64_t* bar,
                                               uint32_t parity) {
  if (!mbar_wait(bar, parity)) {
    S.cabort = 1;
    atomicOr(P.header + kWsStatus, SPECV_DEV_TIMEOUT);
  }
  consumers_sync();
  return S.cabort == 0;
}

// Final-draw weights of chunk j: the residual (p - q)+ or p, both scaled by
// S_p (w = e_p - (S_p/S_q) e_q clipped at 0, or w = e_p).  Draft chunk j
// lies at the same slice offset: both rows keep their own 16-byte phase.
template <int DT>
__device__ __forceinline__ void draw_weights(const unsigned char* bp, const unsigned char* bq,
                                             const SliceGeo& gp, const SliceGeo& gq, int j,
                                             bool residual, float Mp, float Mq, float sT, float r,
                                             float* w) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerChunk;
  float vp[CH], vq[CH];
  E::unpack(reinterpret_cast<const uint4*>(bp)[j], vp);
  const int i0 = chunk_base<DT>(gp, j);
  if (residual) {
    if (gq.h == gp.h) {
      E::unpack(reinterpret_cast<const uint4*>(bq)[j], vq);
    } else {
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int i = i0 + k;
        float z = -INFINITY;
        if (i >= 0 && i < gp.cnt) {
          const unsigned char* src = bq + gq.h + i * E::kBytes;
          z = DT == SPECV_F32 ? *reinterpret_cast<const float*>(src)
                              : __uint_as_float(static_cast<uint32_t>(
                                    *reinterpret_cast<const unsigned short*>(src)) << 16);
        }
        vq[k] = z;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int i = i0 + k;
    float wk = scaled_exp(vp[k], Mp, sT);
    if (residual) wk = fmaxf(__fmaf_rn(-r, scaled_exp(vq[k], Mq, sT), wk), 0.0f);
    w[k] = (i >= 0 && i < gp.cnt) ? wk : 0.0f;
  }
}

template <int DT>
__device__ void consumer(const Params& P, Ctl& S, unsigned char* dyn, int crank, int C, int tid) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerChunk;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int K = P.K;
  uint32_t x2_phase = 0;   // bit (2 * parity + attempt)

  for (int k = 0;; ++k) {
    const int s = k % P.stages;
    const uint32_t ph = static_cast<uint32_t>(k / P.stages) & 1u;
    const int xp = k & 1;
    const uint32_t xph = static_cast<uint32_t>(k >> 1) & 1u;
    if (!consumers_wait(S, P, &S.full[s], ph)) break;
    const Meta m = S.cmeta[s];
    if (m.u < 0) break;
    if (tid == 0) {
      if (C > 1) mbar_arrive_expect_tx(&S.x1_bar[xp], (C - 1) * sizeof(Part));
      else mbar_arrive(&S.x1_bar[xp]);
    }
    const bool greedy = (m.T == 0.0f);
    const bool has_q = !greedy && m.t < m.n;
    const unsigned char* bp = dyn + static_cast<size_t>(s) * P.stage_bytes;
    const unsigned char* bq = bp + P.slice_bytes;
    const size_t trow = static_cast<size_t>(m.b) * (K + 1) + m.t;
    const size_t drow = static_cast<size_t>(m.b) * K + m.t;
    const SliceGeo gp = slice_geo<DT>(P, P.target, trow, crank);
    const SliceGeo gq = has_q ? slice_geo<DT>(P, P.draft, drow, crank) : gp;
    const bool same_phase = gq.h == gp.h;
    const float sT = greedy ? 0.0f : __fdiv_rn(kLog2e, m.T);
    float* rs = P.row_stats ? P.row_stats + (static_cast<size_t>(m.b) * (K + 1) + m.t) * 8 : nullptr;

    if (greedy) {
      // ---- argmax, lowest index on ties --------------------------------
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int j = tid; j < gp.nch; j += kConsumers) {
        const uint4 raw = reinterpret_cast<const uint4*>(bp)[j];
        const bool full = chunk_full<DT>(gp, j);
        if (full && !(E::chunk_max(raw) > bv)) continue;   // no new maximum here
        float v[CH];
        E::unpack(raw, v);
        const int i0 = chunk_base<DT>(gp, j);
#pragma unroll
        for (int q = 0; q < CH; ++q) {
          const int i = i0 + q;
          if (i >= 0 && i < gp.cnt && better(v[q], gp.e0 + i, bv, bi)) { bv = v[q]; bi = gp.e0 + i; }
        }
      }
      warp_argmax(bv, bi);
      if (lane == 0) S.red[warp] = make_float4(bv, __int_as_float(bi), 0.0f, 0.0f);
      consumers_sync();
      if (warp == 0) {
        float v = lane < kConsumerWarps ? S.red[lane].x : -INFINITY;
        int i = lane < kConsumerWarps ? __float_as_int(S.red[lane].y) : INT_MAX;
        warp_argmax(v, i);
        Part part;
        part.a = make_float4(v, __int_as_float(i), 0.0f, 0.0f);
        part.b = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        send_part(S, xp, crank, C, lane, part);
      }
      if (!consumers_wait(S, P, &S.x1_bar[xp], xph)) break;
      float gv = -INFINITY;
      int g = INT_MAX;
      for (int c = 0; c < C; ++c) {
        const float v = S.x1[xp][c].a.x;
        const int i = __float_as_int(S.x1[xp][c].a.y);
        if (better(v, i, gv, g)) { gv = v; g = i; }
      }
      if (crank == 0 && tid == 0) {
        int flags = (m.t < m.n && g == m.x) ? kRecAccept : 0;
        if (g < 0 || g >= P.V) flags |= kRecBad;
        if (rs) {
          rs[0] = gv;
          rs[7] = static_cast<float>(g);
        }
        finish_unit(P, m, g, flags);
      }
    } else {
      // ---- one pass: slice max and sum of exp((z - max)/T) ----------------
      float mp = -INFINITY, sp = 0.0f, mq = -INFINITY, sq = 0.0f;
      for (int j = tid; j < gp.nch; j += kConsumers) {
        const bool full = chunk_full<DT>(gp, j);
        const int i0 = chunk_base<DT>(gp, j);
        {
          const uint4 raw = reinterpret_cast<const uint4*>(bp)[j];
          float v[CH];
          E::unpack(raw, v);
          float cm;
          if (full) {
            cm = E::chunk_max(raw);
          } else {
            cm = -INFINITY;
#pragma unroll
            for (int q = 0; q < CH; ++q) {
              if (i0 + q < 0 || i0 + q >= gp.cnt) v[q] = -INFINITY;
              cm = fmaxf(cm, v[q]);
            }
          }
          if (cm > mp) {
            sp = __fmul_rn(sp, scaled_exp(mp, cm, sT));
            mp = cm;
          }
          if (mp > -INFINITY) {
#pragma unroll
            for (int q = 0; q < CH; ++q) sp = __fadd_rn(sp, scaled_exp(v[q], mp, sT));
          }
        }
        if (has_q) {
          float v[CH];
          float cm = -INFINITY;
          if (same_phase && full) {
            const uint4 raw = reinterpret_cast<const uint4*>(bq)[j];
            E::unpack(raw, v);
            cm = E::chunk_max(raw);
          } else {
#pragma unroll
            for (int q = 0; q < CH; ++q) {
              const int i = i0 + q;
              float z = -INFINITY;
              if (i >= 0 && i < gp.cnt) {
                const unsigned char* src = bq + gq.h + i * E::kBytes;
                z = DT == SPECV_F32 ? *reinterpret_cast<const float*>(src)
                                    : __uint_as_float(static_cast<uint32_t>(
                                          *reinterpret_cast<const unsigned short*>(src)) << 16);
              }
              v[q] = z;
              cm = fmaxf(cm, z);
            }
          }
          if (cm > mq) {
            sq = __fmul_rn(sq, scaled_exp(mq, cm, sT));
            mq = cm;
          }
          if (mq > -INFINITY) {
#pragma unroll
            for (int q = 0; q < CH; ++q) sq = __fadd_rn(sq, scaled_exp(v[q], mq, sT));
          }
        }
      }
      warp_pair(mp, sp, sT);
      warp_pair(mq, sq, sT);
      if (lane == 0) S.red[warp] = make_float4(mp, sp, mq, sq);
      consumers_sync();
      if (warp == 0) {
        float a = -INFINITY, a2 = 0.0f, c2 = -INFINITY, d2 = 0.0f;
        if (lane < kConsumerWarps) {
          const float4 r4 = S.red[lane];
          a = r4.x;
          a2 = r4.y;
          c2 = r4.z;
          d2 = r4.w;
        }
        warp_pair(a, a2, sT);
        warp_pair(c2, d2, sT);
        Part part;
        part.a = make_float4(a, a2, c2, d2);
        float zxp = __int_as_float(0x7fc00000), zxq = __int_as_float(0x7fc00000);
        if (m.t < m.n && m.x >= gp.e0 && m.x < gp.e0 + gp.cnt) {
          const int i = m.x - gp.e0;
          const unsigned char* sp_ = bp + gp.h + i * E::kBytes;
          const unsigned char* sq_ = bq + gq.h + i * E::kBytes;
          if (DT == SPECV_F32) {
            zxp = *reinterpret_cast<const float*>(sp_);
            zxq = *reinterpret_cast<const float*>(sq_);
          } else {
            zxp = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(sp_)) << 16);
            zxq = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(sq_)) << 16);
          }
        }
        part.b = make_float4(zxp, zxq, 0.0f, 0.0f);
        send_part(S, xp, crank, C, lane, part);
      }
      if (!consumers_wait(S, P, &S.x1_bar[xp], xph)) break;

      // ---- combine the cluster's partials (same order in every CTA) -------
      float Mp = -INFINITY, Sp = 0.0f, Mq = -INFINITY, Sq = 0.0f;
      for (int c = 0; c < C; ++c) {
        const float4 a = S.x1[xp][c].a;
        Mp = fmaxf(Mp, a.x);
        Mq = fmaxf(Mq, a.z);
      }
      for (int c = 0; c < C; ++c) {
        const float4 a = S.x1[xp][c].a;
        if (a.x > -INFINITY) Sp = __fadd_rn(Sp, __fmul_rn(a.y, scaled_exp(a.x, Mp, sT)));
        if (a.z > -INFINITY) Sq = __fadd_rn(Sq, __fmul_rn(a.w, scaled_exp(a.z, Mq, sT)));
      }
      // identical in every CTA of the cluster: it steers the exchanges below
      const bool row_ok = isfinite(Mp) && (!has_q || isfinite(Mq));
      bool accept = false;
      float lp = 0.0f, lq = 0.0f;
      if (m.t < m.n) {
        const int ox = m.x / P.slice;
        const float zxp = S.x1[xp][ox].b.x;
        const float zxq = S.x1[xp][ox].b.y;
        lp = __fsub_rn(__fmul_rn(__fsub_rn(zxp, Mp), sT), log2f(Sp));
        lq = __fsub_rn(__fmul_rn(__fsub_rn(zxq, Mq), sT), log2f(Sq));
        accept = __fadd_rn(log2f(m.u_t), lq) < lp;
      }
      const bool want_draw = row_ok && (m.t == m.n || !accept || rs != nullptr);
      if (crank == 0 && tid == 0 && rs) {
        rs[0] = Mp;
        rs[1] = Sp;
        if (m.t < m.n) {
          rs[2] = lp * kLn2;
          rs[3] = Mq;
          rs[4] = Sq;
          rs[5] = lq * kLn2;
        }
      }
      if (!want_draw) {
        if (crank == 0 && tid == 0) {
          int flags = accept ? kRecAccept : 0;
          if (!row_ok) flags |= kRecBad;
          finish_unit(P, m, -1, flags);
        }
      } else {
        // ---- inverse-CDF draw over the on-chip slices -----------------------
        bool residual = m.t < m.n;
        const float u = m.u_draw;
        const float r = __fdiv_rn(Sp, Sq);
        const int ntiles = (gp.nch + kConsumers - 1) / kConsumers;
        int owner = -1;
        float tau_owner = 0.0f, W_report = 0.0f;
        bool aborted = false;
        for (int attempt = 0; attempt < 2; ++attempt) {
          uint64_t* xbar = &S.x2_bar[xp][attempt];
          const int bit = 2 * xp + attempt;
          if (tid == 0) {
            if (C > 1) mbar_arrive_expect_tx(xbar, (C - 1) * 4);
            else mbar_arrive(xbar);
          }
          for (int tile = 0; tile < ntiles; ++tile) {
            const int j = tile * kConsumers + tid;
            float sum = 0.0f;
            if (j < gp.nch) {
              float w[CH];
              draw_weights<DT>(bp, bq, gp, gq, j, residual, Mp, Mq, sT, r, w);
#pragma unroll
              for (int q = 0; q < CH; ++q) sum = __fadd_rn(sum, w[q]);
            }
            const float incl = warp_incl_scan(sum, lane);
            if (lane == 31) S.ws[tile * kConsumerWarps + warp] = incl;
          }
          consumers_sync();
          if (warp == 0) {
            float Wc = 0.0f;
            if (lane == 0) {
              for (int q = 0; q < ntiles * kConsumerWarps; ++q) Wc = __fadd_rn(Wc, S.ws[q]);
              S.x2[xp][attempt][crank] = Wc;
            }
            Wc = __shfl_sync(0xffffffffu, Wc, 0);
            if (lane < C && lane != crank)
              st_async4(peer_addr(&S.x2[xp][attempt][crank], lane), peer_addr(xbar, lane),
                        __float_as_uint(Wc));
          }
          const bool ok = consumers_wait(S, P, xbar, (x2_phase >> bit) & 1u);
          x2_phase ^= 1u << bit;
          if (!ok) {
            aborted = true;
            break;
          }
          // the owning slice: cumulative sums in rank order
          float W = 0.0f;
          for (int c = 0; c < C; ++c) W = __fadd_rn(W, S.x2[xp][attempt][c]);
          const float tau = __fmul_rn(u, W);
          float acc = 0.0f, last_acc = 0.0f;
          int own = -1, last = -1;
          for (int c = 0; c < C; ++c) {
            const float wc = S.x2[xp][attempt][c];
            if (wc > 0.0f) {
              if (own < 0 && __fadd_rn(acc, wc) > tau) {
                own = c;
                tau_owner = __fsub_rn(tau, acc);
              }
              last = c;
              last_acc = acc;
            }
            acc = __fadd_rn(acc, wc);
          }
          if (own < 0 && last >= 0) {
            own = last;
            tau_owner = __fsub_rn(tau, last_acc);
          }
          owner = own;
          if (attempt == 0) W_report = W;
          if (!(residual && !(W > 0.0f))) break;
          residual = false;   // a residual of exactly zero mass: draw from p
        }
        if (aborted) break;
        if (crank == 0 && tid == 0 && rs) rs[6] = __fdiv_rn(W_report, Sp);
        if (owner < 0) {
          if (crank == 0 && tid == 0) finish_unit(P, m, -1, kRecBad);
        } else if (owner == crank) {
          if (tid == 0) {
            float acc = 0.0f, sel_acc = 0.0f, last_acc = 0.0f;
            int sel = -1, last = -1;
            for (int q = 0; q < ntiles * kConsumerWarps; ++q) {
              const float wq = S.ws[q];
              if (wq > 0.0f) {
                if (__fadd_rn(acc, wq) > tau_owner) {
                  sel = q;
                  sel_acc = acc;
                  break;
                }
                last = q;
                last_acc = acc;
              }
              acc = __fadd_rn(acc, wq);
            }
            if (sel < 0) {
              sel = last;
              sel_acc = last_acc;
            }
            if (sel < 0) {
              // no positive weight in the owning slice (cannot happen when its
              // sum is positive): answer the unit as bad rather than never
              finish_unit(P, m, -1, kRecBad);
              S.sel_warp = -1;
            } else {
              S.sel_tile = sel / kConsumerWarps;
              S.sel_warp = sel % kConsumerWarps;
              S.tau_warp = __fsub_rn(tau_owner, sel_acc);
            }
          }
          consumers_sync();
          if (warp == S.sel_warp) {
            const int j = S.sel_tile * kConsumers + tid;
            float w[CH];
            float sum = 0.0f;
            if (j < gp.nch) {
              draw_weights<DT>(bp, bq, gp, gq, j, residual, Mp, Mq, sT, r, w);
#pragma unroll
              for (int q = 0; q < CH; ++q) sum = __fadd_rn(sum, w[q]);
            } else {
#pragma unroll
              for (int q = 0; q < CH; ++q) w[q] = 0.0f;
            }
            const float incl = warp_incl_scan(sum, lane);
            const float tau2 = S.tau_warp;
            const unsigned hit = __ballot_sync(0xffffffffu, sum > 0.0f && incl > tau2);
            const unsigned pos = __ballot_sync(0xffffffffu, sum > 0.0f);
            const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
            const float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (l < 0 && lane == 0) finish_unit(P, m, -1, kRecBad);   // see above
            if (lane == l) {
              const float tau3 = __fsub_rn(tau2, l > 0 ? excl : 0.0f);
              float run = 0.0f;
              int pick = -1, lastq = -1;
#pragma unroll
              for (int q = 0; q < CH; ++q) {
                if (w[q] > 0.0f) {
                  run = __fadd_rn(run, w[q]);
                  if (pick < 0 && run > tau3) pick = q;
                  lastq = q;
                }
              }
              if (pick < 0) pick = lastq;
              const int cand = gp.e0 + chunk_base<DT>(gp, j) + pick;
              int flags = (m.t < m.n && accept) ? kRecAccept : 0;
              if (cand < 0 || cand >= P.V) flags |= kRecBad;
              if (rs) rs[7] = static_cast<float>(cand);
              finish_unit(P, m, cand, flags);
            }
          }
        }
      }
    }
    // ---- release the stage --------------------------------------------------
    consumers_sync();
    if (tid == 0) mbar_arrive(&S.empty[s]);
  }
}

// ---------------------------------------------------------------- kernel

template <int DT>
__global__ void __launch_bounds__(kThreads) verify_kernel(const Params P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int crank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x;

  __shared__ Ctl S;
  extern __shared__ __align__(128) unsigned char dyn[];

  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
      mbar_init(&S.meta_bar[s], 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(&S.x1_bar[p], 1);
      mbar_init(&S.x2_bar[p][0], 1);
      mbar_init(&S.x2_bar[p][1], 1);
    }
    S.pabort = 0;
    S.cabort = 0;
    mbar_init_fence();
  }
  // every CTA's barriers exist before any peer signals them
  cluster.sync();

  if (tid >= kConsumers)
    producer<DT>(P, S, dyn, crank, C, tid - kConsumers);
  else
    consumer<DT>(P, S, dyn, crank, C, tid);

  // no CTA leaves while a peer may still address its shared memory
  cluster.sync();
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(P.header + kWsExit, 1);
    if (prev == static_cast<int>(gridDim.x) - 1) {
      // last CTA of the launch: every ticket is taken; reset for the next call
      P.header[kWsWork] = 0;
      P.header[kWsExit] = 0;
    }
  }
}

// ---------------------------------------------------------------- host side

struct Plan {
  int C;
  int slice;
  int slice_bytes;
  int stage_bytes;
  int stages;
  size_t smem;
  int clusters;
};

int elt_bytes(specv_dtype dt) { return dt == SPECV_BF16 ? 2 : 4; }

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (!v || !*v) return fallback;
  const int x = std::atoi(v);
  return x > 0 ? x : fallback;
}

// Per-device kernel attributes (once) and the number of clusters of C CTAs
// with `smem` dynamic shared memory that fit on the GPU at once.
template <int DT>
cudaError_t max_clusters(int C, size_t smem, int* out) {
  static std::mutex mu;
  static int dev_done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!dev_done[dev]) {
      int optin = 0;
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - static_cast<int>(sizeof(Ctl)));
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      dev_done[dev] = 1;
    }
  }
  // occupancy answers, cached per (device, cluster size, shared memory)
  struct Entry { int dev, C; size_t smem; int clusters; };
  static Entry cache[32];
  static int cached = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < cached; ++i)
      if (cache[i].dev == dev && cache[i].C == C && cache[i].smem == smem) {
        *out = cache[i].clusters;
        return cudaSuccess;
      }
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaOccupancyMaxActiveClusters(out, verify_kernel<DT>, &cfg);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (cached < 32) cache[cached++] = Entry{dev, C, smem, *out};
  return cudaSuccess;
}

// Cluster size, slice and stage ring for a vocabulary size and dtype.
// SPECV_SLICE_BYTES and SPECV_STAGES override the defaults (tuning only).
bool make_plan(int V, specv_dtype dt, bool with_draft, Plan* plan) {
  const int eb = elt_bytes(dt);
  const int per_chunk = kChunkBytes / eb;
  const long long row_bytes = static_cast<long long>(V) * eb;
  const int target = env_int("SPECV_SLICE_BYTES", dt == SPECV_BF16 ? 16384 : 32768);
  long long C = (row_bytes + target - 1) / target;
  if (C < 1) C = 1;
  if (C > kMaxCluster) C = kMaxCluster;
  long long slice = (V + C - 1) / C;
  slice = (slice + per_chunk - 1) / per_chunk * per_chunk;
  if (slice * eb > kSliceMaxBytes) return false;
  C = (V + slice - 1) / slice;
  const int slice_bytes = static_cast<int>((slice * eb + 16 + 127) / 128 * 128);
  const int stage_bytes = slice_bytes * (with_draft ? 2 : 1);
  int stages = env_int("SPECV_STAGES", 0);
  if (stages == 0) {
    stages = (64 * 1024) / stage_bytes;
    if (stages < 2) stages = 2;
  }
  if (stages > kMaxStages) stages = kMaxStages;
  if (static_cast<size_t>(stages) * stage_bytes > 200 * 1024) stages = (200 * 1024) / stage_bytes;
  if (stages < 1) return false;
  plan->C = static_cast<int>(C);
  plan->slice = static_cast<int>(slice);
  plan->slice_bytes = slice_bytes;
  plan->stage_bytes = stage_bytes;
  plan->stages = stages;
  plan->smem = static_cast<size_t>(stages) * stage_bytes;
  return true;
}

size_t ws_header_bytes() { return 16; }
size_t ws_counter_bytes(int B) { return (static_cast<size_t>(B) * 4 + 15) / 16 * 16; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

specv_status launch(const void* target, const void* draft, specv_dtype dtype,
                    const int32_t* draft_tokens, const int32_t* draft_len,
                    const float* temperature, const float* uniforms,
                    const float* uniforms_resample, int B, int K, int V, int32_t* accepted_len,
                    int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                    float* row_stats, cudaStream_t stream) {
  if (!target || !draft_tokens || !temperature || !uniforms || !uniforms_resample ||
      !accepted_len || !out_tokens || !workspace)
    return SPECV_ERR_INVALID_ARG;
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || V < 1) return SPECV_ERR_INVALID_ARG;
  if (B > SPECV_MAX_BATCH || K > SPECV_MAX_DRAFT || V > specv_max_vocab(dtype))
    return SPECV_ERR_UNSUPPORTED;
  const size_t eb = static_cast<size_t>(elt_bytes(dtype));
  if (!aligned(target, eb) || (draft && !aligned(draft, eb)) || !aligned(draft_tokens, 4) ||
      (draft_len && !aligned(draft_len, 4)) || !aligned(temperature, 4) ||
      !aligned(uniforms, 4) || !aligned(uniforms_resample, 4) || !aligned(accepted_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(workspace, 16) || (row_stats && !aligned(row_stats, 4)))
    return SPECV_ERR_INVALID_ARG;
  if (workspace_bytes < specv_workspace_bytes(B, K)) return SPECV_ERR_WORKSPACE;

  Plan plan;
  if (!make_plan(V, dtype, draft != nullptr, &plan)) return SPECV_ERR_UNSUPPORTED;
  int active = 0;
  cudaError_t e = dtype == SPECV_BF16 ? max_clusters<SPECV_BF16>(plan.C, plan.smem, &active)
                                      : max_clusters<SPECV_F32>(plan.C, plan.smem, &active);
  if (e != cudaSuccess || active < 1) return SPECV_ERR_CUDA;
  const long long units = static_cast<long long>(B) * (K + 1);
  plan.clusters = static_cast<int>(units < active ? units : active);

  Params P;
  P.target = target;
  P.draft = draft;
  P.draft_tokens = draft_tokens;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.uniforms = uniforms;
  P.uniforms_resample = uniforms_resample;
  P.B = B;
  P.K = K;
  P.V = V;
  P.units = static_cast<int>(units);
  P.slice = plan.slice;
  P.slice_bytes = plan.slice_bytes;
  P.stage_bytes = plan.stage_bytes;
  P.stages = plan.stages;
  P.accepted_len = accepted_len;
  P.out_tokens = out_tokens;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  P.header = reinterpret_cast<int32_t*>(ws);
  P.counters = reinterpret_cast<int32_t*>(ws + ws_header_bytes());
  P.records = reinterpret_cast<int2*>(ws + ws_header_bytes() + ws_counter_bytes(B));
  P.row_stats = row_stats;

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(plan.C * plan.clusters), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(plan.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = dtype == SPECV_BF16 ? cudaLaunchKernelEx(&cfg, verify_kernel<SPECV_BF16>, P)
                          : cudaLaunchKernelEx(&cfg, verify_kernel<SPECV_F32>, P);
  return e == cudaSuccess ? SPECV_OK : SPECV_ERR_CUDA;
}

size_t pad256(size_t x) { return (x + 255) / 256 * 256; }

// ---------------------------------------------------------------- no-allocation scratch
//
// Scratch for spec_verify_sample_noalloc: the same layout as a caller's
// workspace (header, per-request counters, per-unit records), sized for
// SPECV_NOALLOC_MAX_BATCH requests and SPECV_NOALLOC_MAX_UNITS units.  It is
// a module-scope device array, so every GPU that loads this library holds it
// until the process exits, and every call on a device shares it.
constexpr size_t kNoAllocScratchBytes =
    (16 + 4 * static_cast<size_t>(SPECV_NOALLOC_MAX_BATCH) + 8 * static_cast<size_t>(SPECV_NOALLOC_MAX_UNITS) +
     255) / 256 * 256;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol's name is only a host-side handle, so the address is looked up
// once per device with cudaGetSymbolAddress (with that device current) and
// cached.
cudaError_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

// ---------------------------------------------------------------- C ABI

extern "C" {

int specv_version(void) { return 100; }

int specv_max_vocab(specv_dtype dtype) {
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return 0;
  return kMaxCluster * (kSliceMaxBytes / elt_bytes(dtype));
}

const char* specv_status_string(specv_status status) {
  switch (status) {
    case SPECV_OK: return "ok";
    case SPECV_ERR_INVALID_ARG: return "invalid argument";
    case SPECV_ERR_UNSUPPORTED: return "unsupported shape";
    case SPECV_ERR_WORKSPACE: return "workspace too small";
    case SPECV_ERR_CUDA: return "CUDA error";
    case SPECV_ERR_BAD_INPUT: return "bad input data flagged on the device";
  }
  return "unknown status";
}

size_t specv_workspace_bytes(int B, int K) {
  if (B < 1 || K < 1 || B > SPECV_MAX_BATCH || K > SPECV_MAX_DRAFT) return 0;
  return ws_header_bytes() + ws_counter_bytes(B) + static_cast<size_t>(B) * (K + 1) * 8;
}

specv_status specv_workspace_init(void* workspace, size_t workspace_bytes, specv_stream_t stream) {
  if (!workspace || !aligned(workspace, 16) || workspace_bytes == 0) return SPECV_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SPECV_OK
             : SPECV_ERR_CUDA;
}

specv_status spec_verify_sample(const void* target_logits, const void* draft_logits,
                                specv_dtype dtype, const int32_t* draft_tokens,
                                const int32_t* draft_len, const float* temperature,
                                const float* uniforms, const float* uniforms_resample, int B,
                                int K, int V, int32_t* accepted_len, int32_t* out_tokens,
                                void* workspace, size_t workspace_bytes, specv_stream_t stream) {
  return launch(target_logits, draft_logits, dtype, draft_tokens, draft_len, temperature, uniforms,
                uniforms_resample, B, K, V, accepted_len, out_tokens, workspace, workspace_bytes,
                nullptr, reinterpret_cast<cudaStream_t>(stream));
}

specv_status spec_verify_sample_debug(const void* target_logits, const void* draft_logits,
                                      specv_dtype dtype, const int32_t* draft_tokens,
                                      const int32_t* draft_len, const float* temperature,
                                      const float* uniforms, const float* uniforms_resample,
                                      int B, int K, int V, int32_t* accepted_len,
                                      int32_t* out_tokens, void* workspace,
                                      size_t workspace_bytes, float* row_stats,
                                      specv_stream_t stream) {
  if (!row_stats) return SPECV_ERR_INVALID_ARG;
  return launch(target_logits, draft_logits, dtype, draft_tokens, draft_len, temperature, uniforms,
                uniforms_resample, B, K, V, accepted_len, out_tokens, workspace, workspace_bytes,
                row_stats, reinterpret_cast<cudaStream_t>(stream));
}

specv_status specv_read_device_status(void* workspace, size_t workspace_bytes, int32_t* status,
                                      specv_stream_t stream) {
  if (!workspace || !status || workspace_bytes < ws_header_bytes()) return SPECV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SPECV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPECV_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof word, s) != cudaSuccess) return SPECV_ERR_CUDA;
  *status = word;
  return word ? SPECV_ERR_BAD_INPUT : SPECV_OK;
}

size_t specv_host_staging_bytes(int B, int K, int V, specv_dtype dtype, int with_draft) {
  if (B < 1 || K < 1 || V < 1 || (dtype != SPECV_F32 && dtype != SPECV_BF16)) return 0;
  const size_t eb = static_cast<size_t>(elt_bytes(dtype));
  size_t total = pad256(static_cast<size_t>(B) * (K + 1) * V * eb);
  if (with_draft) total += pad256(static_cast<size_t>(B) * K * V * eb);
  total += pad256(static_cast<size_t>(B) * K * 4);        // draft_tokens
  total += pad256(static_cast<size_t>(B) * 4);            // draft_len
  total += pad256(static_cast<size_t>(B) * 4);            // temperature
  total += pad256(static_cast<size_t>(B) * (K + 1) * 4);  // uniforms
  total += pad256(static_cast<size_t>(B) * 4);            // uniforms_resample
  total += pad256(static_cast<size_t>(B) * 4);            // accepted_len
  total += pad256(static_cast<size_t>(B) * (K + 1) * 4);  // out_tokens
  return total;
}

specv_status spec_verify_sample_host(const void* target_logits, const void* draft_logits,
                                     specv_dtype dtype, const int32_t* draft_tokens,
                                     const int32_t* draft_len, const float* temperature,
                                     const float* uniforms, const float* uniforms_resample,
                                     int B, int K, int V, int32_t* accepted_len,
                                     int32_t* out_tokens, void* staging, size_t staging_bytes,
                                     void* workspace, size_t workspace_bytes,
                                     specv_stream_t stream) {
  if (!target_logits || !draft_tokens || !temperature || !uniforms || !uniforms_resample ||
      !accepted_len || !out_tokens || !staging || !aligned(staging, 256))
    return SPECV_ERR_INVALID_ARG;
  const size_t need = specv_host_staging_bytes(B, K, V, dtype, draft_logits != nullptr);
  if (need == 0) return SPECV_ERR_INVALID_ARG;
  if (staging_bytes < need) return SPECV_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t eb = static_cast<size_t>(elt_bytes(dtype));
  unsigned char* cur = static_cast<unsigned char*>(staging);
  auto take = [&](size_t bytes) {
    unsigned char* p = cur;
    cur += pad256(bytes);
    return p;
  };
  auto h2d = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  const size_t tb = static_cast<size_t>(B) * (K + 1) * V * eb;
  const size_t db = static_cast<size_t>(B) * K * V * eb;
  void* d_t = take(tb);
  void* d_d = draft_logits ? take(db) : nullptr;
  int32_t* d_tok = reinterpret_cast<int32_t*>(take(static_cast<size_t>(B) * K * 4));
  int32_t* d_len = reinterpret_cast<int32_t*>(take(static_cast<size_t>(B) * 4));
  float* d_T = reinterpret_cast<float*>(take(static_cast<size_t>(B) * 4));
  float* d_u = reinterpret_cast<float*>(take(static_cast<size_t>(B) * (K + 1) * 4));
  float* d_ur = reinterpret_cast<float*>(take(static_cast<size_t>(B) * 4));
  int32_t* d_acc = reinterpret_cast<int32_t*>(take(static_cast<size_t>(B) * 4));
  int32_t* d_out = reinterpret_cast<int32_t*>(take(static_cast<size_t>(B) * (K + 1) * 4));
  bool ok = h2d(d_t, target_logits, tb);
  if (draft_logits) ok = ok && h2d(d_d, draft_logits, db);
  ok = ok && h2d(d_tok, draft_tokens, static_cast<size_t>(B) * K * 4);
  if (draft_len) ok = ok && h2d(d_len, draft_len, static_cast<size_t>(B) * 4);
  ok = ok && h2d(d_T, temperature, static_cast<size_t>(B) * 4);
  ok = ok && h2d(d_u, uniforms, static_cast<size_t>(B) * (K + 1) * 4);
  ok = ok && h2d(d_ur, uniforms_resample, static_cast<size_t>(B) * 4);
  if (!ok) return SPECV_ERR_CUDA;
  specv_status st = launch(d_t, d_d, dtype, d_tok, draft_len ? d_len : nullptr, d_T, d_u, d_ur, B,
                           K, V, d_acc, d_out, workspace, workspace_bytes, nullptr, s);
  if (st != SPECV_OK) return st;
  if (cudaMemcpyAsync(accepted_len, d_acc, static_cast<size_t>(B) * 4, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(out_tokens, d_out, static_cast<size_t>(B) * (K + 1) * 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? SPECV_OK : SPECV_ERR_CUDA;
}

specv_status specv_launch_plan(int B, int K, int V, specv_dtype dtype, int with_draft,
                               int32_t* out) {
  if (!out || B < 1 || K < 1 || V < 1 || (dtype != SPECV_F32 && dtype != SPECV_BF16))
    return SPECV_ERR_INVALID_ARG;
  if (B > SPECV_MAX_BATCH || K > SPECV_MAX_DRAFT || V > specv_max_vocab(dtype))
    return SPECV_ERR_UNSUPPORTED;
  Plan plan;
  if (!make_plan(V, dtype, with_draft != 0, &plan)) return SPECV_ERR_UNSUPPORTED;
  int active = 0;
  const cudaError_t e = dtype == SPECV_BF16 ? max_clusters<SPECV_BF16>(plan.C, plan.smem, &active)
                                            : max_clusters<SPECV_F32>(plan.C, plan.smem, &active);
  if (e != cudaSuccess) return SPECV_ERR_CUDA;
  const long long units = static_cast<long long>(B) * (K + 1);
  out[0] = plan.C;
  out[1] = plan.slice;
  out[2] = plan.stages;
  out[3] = static_cast<int32_t>(units < active ? units : active);
  out[4] = static_cast<int32_t>(plan.smem);
  out[5] = kThreads;
  return SPECV_OK;
}

specv_status spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                        specv_dtype dtype, const int32_t* draft_tokens,
                                        const int32_t* draft_len, const float* temperature,
                                        const float* uniforms, const float* uniforms_resample,
                                        int B, int K, int V, int32_t* accepted_len,
                                        int32_t* out_tokens, specv_stream_t stream) {
  if (B < 1 || K < 1 || K > SPECV_MAX_DRAFT) return SPECV_ERR_INVALID_ARG;
  if (B > SPECV_NOALLOC_MAX_BATCH ||
      static_cast<long long>(B) * (K + 1) > SPECV_NOALLOC_MAX_UNITS)
    return SPECV_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return SPECV_ERR_CUDA;
  const size_t bytes = specv_workspace_bytes(B, K);
  // The array keeps the previous call's contents: zero the status word and
  // the arrival counters this call relies on.
  if (cudaMemsetAsync(scratch, 0, bytes, s) != cudaSuccess) return SPECV_ERR_CUDA;
  return launch(target_logits, draft_logits, dtype, draft_tokens, draft_len, temperature, uniforms,
                uniforms_resample, B, K, V, accepted_len, out_tokens, scratch, bytes, nullptr, s);
}

}  // extern "C"
