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
// Work is split into tiles of one 16 KB chunk of one row.  Groups of four
// consecutive chunks of a row are dealt round-robin, in request-major order,
// to a grid of persistent CTAs.  Each CTA has three roles:
//   * a producer warp streams each of its tiles' chunk(s) into a ring of
//     shared-memory stages with TMA bulk copies (full / empty mbarriers);
//   * eight consumer warps reduce a stats tile to a partial - the chunk's
//     maximum and sum of exp((z - max)/T), or its argmax at T = 0, plus the
//     drafted token's logit if the chunk holds it - or, for a draw tile, to
//     per-warp prefix sums of the final-draw weights;
//   * a control warp counts finished tiles per request (acq_rel atomics).
//     The CTA that finishes a request's last stats tile combines the
//     request's partials, runs the left-to-right accept test and publishes
//     the decision; for a sampled request the final row (a rejected
//     position's residual (p - q)+, or the bonus position's p) is then read
//     again as draw tiles, each chunk group owned by a fixed CTA that polls
//     for the decision.  The CTA that finishes the last draw tile locates the
//     drawn token from the per-warp sums, re-reading one 32-vector segment,
//     and writes the outputs.
// No CTA waits for another: every wait is on this CTA's own mbarriers and is
// bounded in time, with a status bit on timeout.  Each needed logit is read
// from HBM once; the final row of a sampled request is read a second time,
// normally from L2, because tickets run request by request.

#include <cuda/atomic>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "specverify.h"

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kControlWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumers + 64;
constexpr int kChunkBytes = 16384;                        // one tile of one row
constexpr int kVecs = kChunkBytes / 16 + 1;               // 16-byte vectors incl. phase
constexpr int kSweeps = (kVecs + kConsumers - 1) / kConsumers;
constexpr int kParts = kSweeps * kConsumerWarps;          // per chunk, per weight mode
constexpr int kSlotBytes = kChunkBytes + 128;
constexpr int kStageBytes = 2 * kSlotBytes;               // target chunk + draft chunk
constexpr int kMaxStages = 6;
constexpr int kMailbox = 32;
constexpr int kGroup = 4;                                 // chunks per dealt group
constexpr int kCtlBuf = 2048;                             // control-warp staging (floats)
constexpr int kRunMax = 8;                                // event groups per control pass
constexpr int kMaxChunks = 128;                           // per row
constexpr long long kWaitLimitCycles = 4000000000ll;      // ~2 s at 2 GHz
constexpr uint32_t kSuspendHintNs = 20000;

// workspace header words, one 128-byte line each
constexpr int kHStatus = 0, kHExit = 32, kHEpoch = 64;
constexpr int kHeaderBytes = 512;

// per-request decision state: (call tag << 2) | value
constexpr int kStateDraws = 1, kStateNone = 2;

// tile kinds and control events
constexpr int kTileSentinel = 0, kTileStats = 1, kTileDraw = 2;
constexpr int kEvSentinel = 0, kEvStats = 1, kEvDraw = 2;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Per-request state in the workspace (64 bytes).
struct Req {
  int stats_done;   // stats tiles finished
  int draw_done;    // draw tiles finished
  int j;            // accepted drafts
  int t_f;          // row of the final draw
  int residual;     // final draw from (p - q)+ (else from p)
  int state;        // decision, tagged with the call (kStateDraws / kStateNone)
  int pad1, pad2;
  float u;          // uniform of the final draw
  float Mp, Mq;     // row maxima (raw logits)
  float sT;         // log2(e) / T
  float ratio;      // S_p / S_q
  float Sp, Sq;
  float pad3;
};

struct Params {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  const float* uniforms;
  const float* uniforms_resample;
  int B, K, V;
  int R;            // rows per request in the ticket space: K+1 target, K draft
  int NC;           // chunks per row
  int NG;           // chunk groups per row
  int CE;           // elements per chunk
  int stages;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t* header;
  Req* req;         // [B]
  float2* part;     // [B][R][NC] stats partials
  float* zx;        // [B][R] logit of the drafted token in each row
  float* dpart;     // [B][NC][2][kParts] draw partial sums (mode 0: final weights, 1: p)
  float* row_stats; // [B][K+1][8] or null
};

// One tile as the producer hands it to the consumers (64 bytes).
struct __align__(16) Tile {
  int kind, b, r, c;
  int x, greedy, t, residual;
  float sT, Mp, Mq, ratio;
  int pad[4];
};

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t mb_full[kMailbox];
  uint64_t mb_empty[kMailbox];
  Tile tile[kMaxStages];
  int2 mb[kMailbox];
  float4 wpart[kMaxStages][kConsumerWarps];   // per-warp partials of a stats tile
  int done_cnt[kMaxStages];                     // consumer warps finished with a stage
  int mb_head;                                  // next mailbox slot to fill
  alignas(16) float cbuf[kCtlBuf];   // control warp: staged partials (read as float2)
  float ctot[kMaxChunks];       // control warp: chunk totals
  int run_kind[kRunMax], run_b[kRunMax], run_cnt[kRunMax];
  uint32_t tag;     // this call's tag for request states
};

// ---------------------------------------------------------------- elements

template <int DT> struct Elt;
template <> struct Elt<SPECV_F32> {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
  __device__ static void unpack(uint4 raw, float v[4]) {
    v[0] = __uint_as_float(raw.x);
    v[1] = __uint_as_float(raw.y);
    v[2] = __uint_as_float(raw.z);
    v[3] = __uint_as_float(raw.w);
  }
  __device__ static float vec_max(uint4 raw) {
    return fmaxf(fmaxf(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                 fmaxf(__uint_as_float(raw.z), __uint_as_float(raw.w)));
  }
  __device__ static float load(const unsigned char* p) { return *reinterpret_cast<const float*>(p); }
  // running elementwise max of vectors, and its final value
  struct MaxAcc {
    float a = -INFINITY, b = -INFINITY;
    __device__ void add(uint4 raw) {
      a = fmaxf(a, fmaxf(__uint_as_float(raw.x), __uint_as_float(raw.y)));
      b = fmaxf(b, fmaxf(__uint_as_float(raw.z), __uint_as_float(raw.w)));
    }
    __device__ float value() const { return fmaxf(a, b); }
  };
  __device__ static float ldg(const unsigned char* p) {
    return __ldg(reinterpret_cast<const float*>(p));
  }
  __device__ static void copy1(unsigned char* dst, const unsigned char* src) {
    *reinterpret_cast<float*>(dst) = __ldg(reinterpret_cast<const float*>(src));
  }
};
template <> struct Elt<SPECV_BF16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
  __device__ static void unpack(uint4 raw, float v[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  // Maximum of 8 bf16 values with packed bf16x2 max, then widened.
  __device__ static float vec_max(uint4 raw) {
    uint32_t m01, m23, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m01) : "r"(raw.x), "r"(raw.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m23) : "r"(raw.z), "r"(raw.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m01), "r"(m23));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ static float load(const unsigned char* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
  }
  // running elementwise max of vectors in packed bf16x2, and its value
  struct MaxAcc {
    uint32_t w[4] = {0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u};   // -inf
    __device__ void add(uint4 raw) {
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[0]) : "r"(raw.x));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[1]) : "r"(raw.y));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[2]) : "r"(raw.z));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[3]) : "r"(raw.w));
    }
    __device__ float value() const {
      return vec_max(make_uint4(w[0], w[1], w[2], w[3]));
    }
  };
  __device__ static float ldg(const unsigned char* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)))
                           << 16);
  }
  __device__ static void copy1(unsigned char* dst, const unsigned char* src) {
    *reinterpret_cast<unsigned short*>(dst) = __ldg(reinterpret_cast<const unsigned short*>(src));
  }
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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

// Non-blocking test of phase `parity` (acquire on success).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of the barrier; gives up after kWaitLimitCycles.
// Called by one thread of a group: the others wait on a hardware barrier,
// so polling never takes issue slots from the warps doing the work; the
// poller sleeps between polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (ns < 256) ns <<= 1;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// Whole warp: lane 0 waits, the other lanes take the phase afterwards.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_wait(bar, parity);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_test(bar, parity);
  return ok != 0;
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

// 2^x on the MUFU unit (PTX ex2.approx.ftz.f32); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp((z - m)/T) as 2^((z - m) * log2(e)/T), the argument formed from the
// exact difference to the reference m.
__device__ __forceinline__ float scaled_exp(float z, float m, float sT) {
  return ex2(__fmul_rn(__fsub_rn(z, m), sT));
}

__device__ __forceinline__ float temp_scale(float T) { return __fdiv_rn(kLog2e, T); }

using AtomicInt = cuda::atomic_ref<int, cuda::thread_scope_device>;

// ---------------------------------------------------------------- reductions

// Online (max, sum of exp) pairs: the sum is relative to the max.
__device__ __forceinline__ void pair_combine(float& m, float& s, float om, float os, float sT) {
  const float M = fmaxf(m, om);
  if (M == -INFINITY) {
    m = M;
    s = 0.0f;
    return;
  }
  s = __fadd_rn(__fmul_rn(s, scaled_exp(m, M, sT)), __fmul_rn(os, scaled_exp(om, M, sT)));
  m = M;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Warp-wide (max, sum of exp) from per-lane pairs relative to each lane's
// max: the max first, then every lane rescales its sum once, then a sum.
__device__ __forceinline__ void warp_max_sum(float& m, float& s, float sT) {
  const float M = warp_max(m);
  const float sc = (m > -INFINITY) ? __fmul_rn(s, scaled_exp(m, M, sT)) : 0.0f;
  s = warp_sum(sc);
  m = M;
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
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

// ---------------------------------------------------------------- chunks

// Where chunk c of a row sits: elements [e0, e0 + cnt) of the row.  Shared
// memory keeps the row's global 16-byte phase h, so element i of the chunk
// is at byte h + i * elt and vector j covers bytes [16 j, 16 j + 16).
struct Geo {
  int e0, cnt, h, nvec;
};

template <int DT>
__device__ __forceinline__ const unsigned char* row_ptr(const void* base, size_t row, int V) {
  return static_cast<const unsigned char*>(base) + row * static_cast<size_t>(V) * Elt<DT>::kBytes;
}

template <int DT>
__device__ __forceinline__ Geo chunk_geo(const Params& P, const unsigned char* row, int c) {
  using E = Elt<DT>;
  Geo g;
  g.e0 = c * P.CE;
  g.cnt = min(P.CE, P.V - g.e0);
  g.h = static_cast<int>((reinterpret_cast<uintptr_t>(row) + static_cast<size_t>(g.e0) * E::kBytes) & 15);
  g.nvec = (g.h + g.cnt * E::kBytes + 15) / 16;
  return g;
}

template <int DT>
__device__ __forceinline__ int vec_base(const Geo& g, int j) {
  return (16 * j - g.h) / Elt<DT>::kBytes;
}

template <int DT>
__device__ __forceinline__ bool vec_full(const Geo& g, int j) {
  const int i0 = vec_base<DT>(g, j);
  return i0 >= 0 && i0 + Elt<DT>::kPerVec <= g.cnt;
}

// Values of vector j of a chunk held in shared memory; lanes outside the
// chunk read as -inf.
template <int DT>
__device__ __forceinline__ void smem_vec(const unsigned char* buf, const Geo& g, int j, float* v) {
  using E = Elt<DT>;
  E::unpack(reinterpret_cast<const uint4*>(buf)[j], v);
  if (!vec_full<DT>(g, j)) {
    const int i0 = vec_base<DT>(g, j);
#pragma unroll
    for (int q = 0; q < E::kPerVec; ++q)
      if (i0 + q < 0 || i0 + q >= g.cnt) v[q] = -INFINITY;
  }
}

// Final-draw weights of one vector: mode 0 = the residual (p - q)+ (or p at
// the bonus position), mode 1 = p; both scaled by S_p.
template <int DT>
__device__ __forceinline__ void vec_weights(const float* vp, const float* vq, bool residual,
                                            float Mp, float Mq, float sT, float ratio, float* w0,
                                            float* w1) {
  constexpr int CH = Elt<DT>::kPerVec;
#pragma unroll
  for (int q = 0; q < CH; ++q) {
    const float ep = scaled_exp(vp[q], Mp, sT);
    w1[q] = ep;
    w0[q] = residual ? fmaxf(__fmaf_rn(-ratio, scaled_exp(vq[q], Mq, sT), ep), 0.0f) : ep;
  }
}

// ---------------------------------------------------------------- requests

__device__ int request_len(const Params& P, int b) {
  return P.draft_len ? __ldg(P.draft_len + b) : P.K;
}

// Stats tiles a valid request needs: target rows t <= n, draft rows t < n
// when sampled, every chunk.
__device__ __forceinline__ int request_tiles(const Params& P, int n, float T) {
  return ((n + 1) + (T > 0.0f ? n : 0)) * P.NC;
}

// Writes a finished request's outputs and returns its counters to zero.
__device__ void finish_request(const Params& P, int b, int j, int tok, int lane) {
  const int K = P.K;
  int32_t* out = P.out_tokens + static_cast<size_t>(b) * (K + 1);
  for (int s = lane; s <= K; s += 32) {
    int v = -1;
    if (j < 0) v = -1;
    else if (s < j) v = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + s);
    else if (s == j) v = tok;
    out[s] = v;
  }
  if (lane == 0) {
    P.accepted_len[b] = j;
    P.req[b].stats_done = 0;
    P.req[b].draw_done = 0;
  }
  __syncwarp();
}

// Publishes request b's decision for the producers that own its draw tiles.
__device__ __forceinline__ void set_state(const Params& P, int b, uint32_t tag, int v) {
  AtomicInt(P.req[b].state).store(static_cast<int>((tag << 2) | static_cast<uint32_t>(v)),
                                  cuda::memory_order_release);
}

__device__ void finish_bad(const Params& P, int b, int bits, int lane, uint32_t tag) {
  if (lane == 0) {
    atomicOr(P.header + kHStatus, bits);
    set_state(P, b, tag, kStateNone);
  }
  finish_request(P, b, -1, -1, lane);
}

// ---------------------------------------------------------------- producer

// Copies one chunk into shared memory: the 16-byte-aligned interior by one
// bulk copy (issued later by lane 0), the unaligned head and tail by the
// lanes.  Returns the bulk byte count.
template <int DT>
__device__ uint32_t stage_chunk(const Params& P, const unsigned char* row, int c,
                                unsigned char* dst, int lane, const unsigned char** bulk_src,
                                unsigned char** bulk_dst) {
  using E = Elt<DT>;
  const Geo g = chunk_geo<DT>(P, row, c);
  const unsigned char* gsrc = row + static_cast<size_t>(g.e0) * E::kBytes;
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
  const int nhead = static_cast<int>((head_end - s0) / E::kBytes);
  const int ntail = static_cast<int>((s1 - tail_begin) / E::kBytes);
  for (int i = lane; i < nhead + ntail; i += 32) {
    const uintptr_t off = i < nhead ? static_cast<uintptr_t>(i) * E::kBytes
                                    : (tail_begin - s0) + static_cast<uintptr_t>(i - nhead) * E::kBytes;
    E::copy1(dst + g.h + off, gsrc + off);
  }
  return bulk;
}

// Stages one tile into the ring (waits, bounded, for a free stage).
template <int DT>
__device__ bool issue_tile(const Params& P, Ctl& S, unsigned char* dyn, int lane, int& k,
                           const Tile& tl) {
  const int K = P.K;
  const int s = k % P.stages;
  const uint32_t ph = static_cast<uint32_t>(k / P.stages) & 1u;
  if (!warp_wait(&S.empty[s], ph ^ 1u, lane)) return false;
  unsigned char* slot0 = dyn + static_cast<size_t>(s) * kStageBytes;
  const unsigned char *src0 = nullptr, *src1 = nullptr;
  unsigned char *dst0 = nullptr, *dst1 = nullptr;
  uint32_t b0 = 0, b1 = 0;
  if (tl.kind == kTileStats) {
    const bool is_draft = tl.r > K;
    const size_t row = is_draft ? static_cast<size_t>(tl.b) * K + tl.t
                                : static_cast<size_t>(tl.b) * (K + 1) + tl.t;
    const unsigned char* rp = row_ptr<DT>(is_draft ? P.draft : P.target, row, P.V);
    b0 = stage_chunk<DT>(P, rp, tl.c, slot0, lane, &src0, &dst0);
  } else {
    const unsigned char* rp = row_ptr<DT>(P.target, static_cast<size_t>(tl.b) * (K + 1) + tl.t, P.V);
    b0 = stage_chunk<DT>(P, rp, tl.c, slot0, lane, &src0, &dst0);
    if (tl.residual) {
      const unsigned char* rq = row_ptr<DT>(P.draft, static_cast<size_t>(tl.b) * K + tl.t, P.V);
      b1 = stage_chunk<DT>(P, rq, tl.c, slot0 + kSlotBytes, lane, &src1, &dst1);
    }
  }
  if (lane == 0) S.tile[s] = tl;
  __syncwarp();
  if (lane == 0) {
    mbar_arrive_expect_tx(&S.full[s], b0 + b1);
    if (b0) bulk_copy_g2s(dst0, src0, b0, &S.full[s]);
    if (b1) bulk_copy_g2s(dst1, src1, b1, &S.full[s]);
  }
  ++k;
  return true;
}

// Issues the draw tiles this CTA owns.  Draw group D = b * NG + d (chunks
// [4d, 4d + 4) of request b's final row) belongs to CTA D mod grid, so this
// CTA walks D = blockIdx.x + i * grid in request order, from the cursor i,
// issuing the group of every request whose decision is published.  Without
// `blocking` it returns at the first undecided request (a relaxed peek, so
// the producer does not stall); with `blocking` it waits (bounded) for each.
template <int DT>
__device__ bool serve_draws(const Params& P, Ctl& S, unsigned char* dyn, int lane, int& k,
                            long long& di, bool blocking) {
  const int NC = P.NC, NG = P.NG;
  const uint32_t tag = S.tag;
  const long long total = static_cast<long long>(P.B) * NG;
  for (;;) {
    const long long D = blockIdx.x + di * static_cast<long long>(gridDim.x);
    if (D >= total) return true;
    const int b = static_cast<int>(D / NG);
    const int dg = static_cast<int>(D - static_cast<long long>(b) * NG);
    int st = 0;
    if (lane == 0) {
      const int peek = AtomicInt(P.req[b].state).load(cuda::memory_order_relaxed);
      if ((static_cast<uint32_t>(peek) >> 2) == tag) st = peek & 3;
      if (st == 0 && blocking) {
        const long long t0 = clock64();
        for (;;) {
          __nanosleep(200);
          const int v = AtomicInt(P.req[b].state).load(cuda::memory_order_relaxed);
          if ((static_cast<uint32_t>(v) >> 2) == tag) {
            st = v & 3;
            break;
          }
          if (clock64() - t0 > kWaitLimitCycles) {
            st = -1;
            break;
          }
        }
      }
      if (st > 0) AtomicInt(P.req[b].state).load(cuda::memory_order_acquire);   // order the reads below
    }
    st = __shfl_sync(0xffffffffu, st, 0);
    __syncwarp();
    if (st < 0) return false;
    if (st == 0) return true;   // not decided yet: look again later
    if (st == kStateDraws) {
      const Req* q = P.req + b;
      Tile tl;
      tl.kind = kTileDraw;
      tl.b = b;
      tl.r = 0;
      tl.t = __ldcg(&q->t_f);
      tl.residual = __ldcg(&q->residual);
      tl.sT = __ldcg(&q->sT);
      tl.Mp = __ldcg(&q->Mp);
      tl.Mq = __ldcg(&q->Mq);
      tl.ratio = __ldcg(&q->ratio);
      tl.x = -1;
      tl.greedy = 0;
      for (int c = dg * kGroup; c < min(NC, dg * kGroup + kGroup); ++c) {
        tl.c = c;
        if (!issue_tile<DT>(P, S, dyn, lane, k, tl)) return false;
      }
    }
    ++di;
  }
}

// The producer warp: this CTA's stats groups (groups g, g + grid, ... of the
// request-major group space), its draw tiles as their requests are decided,
// then a sentinel.  Requests whose length or temperature is unusable are
// answered by the owner of their first group.
template <int DT>
__device__ void producer(const Params& P, Ctl& S, unsigned char* dyn, int lane) {
  const int K = P.K, NC = P.NC, R = P.R, NG = P.NG;
  const long long total = static_cast<long long>(P.B) * R * NG;
  int k = 0;         // stage uses
  long long di = 0;  // draw cursor
  bool ok = true;
  int mb = -1, mn = 0, mbad = 0;
  float mT = 0.0f;
  for (long long gi = blockIdx.x; gi < total && ok; gi += gridDim.x) {
    const int cg = static_cast<int>(gi % NG);
    const long long br = gi / NG;
    const int r = static_cast<int>(br % R);
    const int b = static_cast<int>(br / R);
    if (b != mb) {
      mb = b;
      mn = request_len(P, b);
      mT = __ldg(P.temperature + b);
      mbad = 0;
      if (mn < 1 || mn > K) mbad = SPECV_DEV_BAD_DRAFT_LEN;
      else if (!(mT >= 0.0f) || isinf(mT)) mbad = SPECV_DEV_BAD_TEMPERATURE;
      else if (mT > 0.0f && P.draft == nullptr) mbad = SPECV_DEV_NO_DRAFT;
    }
    if (mbad) {
      if (r == 0 && cg == 0) finish_bad(P, b, mbad, lane, S.tag);
      continue;
    }
    const bool sampled = mT > 0.0f;
    const bool valid = r <= K ? r <= mn : (sampled && r - (K + 1) < mn);
    if (!valid) continue;   // rows after the draft are never read
    Tile tl;
    tl.kind = kTileStats;
    tl.b = b;
    tl.r = r;
    tl.t = r <= K ? r : r - (K + 1);
    tl.greedy = !sampled;
    tl.x = tl.t < mn ? __ldg(P.draft_tokens + static_cast<size_t>(b) * K + tl.t) : -1;
    tl.sT = sampled ? temp_scale(mT) : 0.0f;
    tl.residual = 0;
    tl.Mp = tl.Mq = tl.ratio = 0.0f;
    for (int c = cg * kGroup; c < min(NC, cg * kGroup + kGroup) && ok; ++c) {
      tl.c = c;
      ok = issue_tile<DT>(P, S, dyn, lane, k, tl);
    }
    if (ok) ok = serve_draws<DT>(P, S, dyn, lane, k, di, false);
  }
  if (ok) ok = serve_draws<DT>(P, S, dyn, lane, k, di, true);
  if (!ok && lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
  // sentinel: the consumers stop at it
  const int s = k % P.stages;
  const uint32_t ph = static_cast<uint32_t>(k / P.stages) & 1u;
  const bool free_slot = warp_wait(&S.empty[s], ph ^ 1u, lane);
  if (lane == 0) {
    if (!free_slot) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
    S.tile[s].kind = kTileSentinel;
    mbar_arrive(&S.full[s]);
  }
}

// ---------------------------------------------------------------- consumers

// Each consumer warp runs on its own: it waits for a stage itself, and no
// block-wide barrier is taken per tile.

// Lane 0 of the posting warp: hands an event to the control warp.  Several
// warps may post; each reserves a mailbox slot with a block-scope atomic.
__device__ __forceinline__ void post_event(Ctl& S, const Params& P, int kind, int b) {
  const int e = atomicAdd_block(&S.mb_head, 1);
  const int slot = e % kMailbox;
  const uint32_t ph = static_cast<uint32_t>(e / kMailbox) & 1u;
  if (!mbar_wait(&S.mb_empty[slot], ph ^ 1u)) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
  S.mb[slot] = make_int2(kind, b);
  mbar_arrive(&S.mb_full[slot]);
}

// Lane 0: counts this warp's finish of the tile in stage s; true for the
// last of the consumer warps (the one that combines and posts).
__device__ __forceinline__ bool last_warp(Ctl& S, int s) {
  __threadfence_block();
  const bool last = atomicAdd_block(&S.done_cnt[s], 1) == kConsumerWarps - 1;
  if (last) {
    S.done_cnt[s] = 0;
    __threadfence_block();
  }
  return last;
}

template <int DT>
__device__ void consumer(const Params& P, Ctl& S, unsigned char* dyn, int tid) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int K = P.K;
  for (int k = 0;; ++k) {
    const int s = k % P.stages;
    const uint32_t ph = static_cast<uint32_t>(k / P.stages) & 1u;
    const bool ok = warp_wait(&S.full[s], ph, lane);
    const Tile tl = S.tile[s];
    if (!ok || tl.kind == kTileSentinel) {
      // the last warp to stop tells the control warp (after every event)
      int last = 0;
      if (lane == 0) last = last_warp(S, s);
      if (__shfl_sync(0xffffffffu, last, 0) && lane == 0) post_event(S, P, kEvSentinel, 0);
      if (!ok && lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
      break;
    }
    const unsigned char* buf0 = dyn + static_cast<size_t>(s) * kStageBytes;
    const unsigned char* buf1 = buf0 + kSlotBytes;

    if (tl.kind == kTileStats) {
      const bool is_draft = tl.r > K;
      const size_t row = is_draft ? static_cast<size_t>(tl.b) * K + tl.t
                                  : static_cast<size_t>(tl.b) * (K + 1) + tl.t;
      const unsigned char* rp = row_ptr<DT>(is_draft ? P.draft : P.target, row, P.V);
      const Geo g = chunk_geo<DT>(P, rp, tl.c);
      // interior vectors [jlo, jhi) hold only chunk elements; at most the
      // first and the last vector are partial and are masked
      const int jlo = g.h > 0 ? 1 : 0;
      const int jhi = max(jlo, (g.h + g.cnt * E::kBytes) / 16);
      const int edge0 = (jlo == 1) ? 0 : -1;                       // thread 0
      const int edge1 = (jhi < g.nvec && jhi != edge0) ? jhi : -1;  // thread 1
      const int my_edge = tid == 0 ? edge0 : (tid == 1 ? edge1 : -1);
      float4 wpart;
      if (tl.greedy) {
        // ---- argmax, lowest index on ties ----------------------------------
        typename E::MaxAcc acc;
        for (int j = jlo + tid; j < jhi; j += kConsumers) acc.add(reinterpret_cast<const uint4*>(buf0)[j]);
        float mx = acc.value();
        if (my_edge >= 0) {
          float v[CH];
          smem_vec<DT>(buf0, g, my_edge, v);
#pragma unroll
          for (int q = 0; q < CH; ++q) mx = fmaxf(mx, v[q]);
        }
        const float W = warp_max(mx);
        // the first element equal to the warp's max, searched only by the
        // lanes whose own maximum it is
        int idx = INT_MAX;
        if (mx == W && W > -INFINITY) {
          if (my_edge == 0) {
            float v[CH];
            smem_vec<DT>(buf0, g, 0, v);
#pragma unroll
            for (int q = CH - 1; q >= 0; --q)
              if (v[q] == W) idx = g.e0 + vec_base<DT>(g, 0) + q;
          }
          for (int j = jlo + tid; j < jhi && idx == INT_MAX; j += kConsumers) {
            float v[CH];
            E::unpack(reinterpret_cast<const uint4*>(buf0)[j], v);
#pragma unroll
            for (int q = CH - 1; q >= 0; --q)
              if (v[q] == W) idx = g.e0 + vec_base<DT>(g, j) + q;
          }
          if (idx == INT_MAX && my_edge > 0) {
            float v[CH];
            smem_vec<DT>(buf0, g, my_edge, v);
#pragma unroll
            for (int q = CH - 1; q >= 0; --q)
              if (v[q] == W) idx = g.e0 + vec_base<DT>(g, my_edge) + q;
          }
        }
        idx = warp_min_int(idx);
        if (!(W > -INFINITY)) idx = g.e0;   // all -inf: the lowest index
        wpart = make_float4(W, __int_as_float(idx), 0.0f, 0.0f);
      } else {
        // ---- one pass: chunk max and sum of exp((z - max)/T) ---------------
        // exponents are fma(z, sT, -c) against c = fl(m sT), m the running
        // max; the rounding of c is taken out once at the end
        const float sT = tl.sT;
        float m = -INFINITY, c = INFINITY, s0 = 0.0f, s1 = 0.0f;
        for (int j = jlo + tid; j < jhi; j += kConsumers) {
          const uint4 raw = reinterpret_cast<const uint4*>(buf0)[j];
          const float cm = E::vec_max(raw);
          if (cm > m) {
            const float cn = __fmul_rn(cm, sT);
            const float f = (m > -INFINITY) ? ex2(__fsub_rn(c, cn)) : 0.0f;
            s0 = __fmul_rn(s0, f);
            s1 = __fmul_rn(s1, f);
            m = cm;
            c = cn;
          }
          float v[CH];
          E::unpack(raw, v);
#pragma unroll
          for (int q = 0; q < CH; q += 2) {
            s0 = __fadd_rn(s0, ex2(__fmaf_rn(v[q], sT, -c)));
            s1 = __fadd_rn(s1, ex2(__fmaf_rn(v[q + 1], sT, -c)));
          }
        }
        if (my_edge >= 0) {
          float v[CH];
          smem_vec<DT>(buf0, g, my_edge, v);
          float cm = -INFINITY;
#pragma unroll
          for (int q = 0; q < CH; ++q) cm = fmaxf(cm, v[q]);
          if (cm > m) {
            const float cn = __fmul_rn(cm, sT);
            const float f = (m > -INFINITY) ? ex2(__fsub_rn(c, cn)) : 0.0f;
            s0 = __fmul_rn(s0, f);
            s1 = __fmul_rn(s1, f);
            m = cm;
            c = cn;
          }
#pragma unroll
          for (int q = 0; q < CH; ++q) s0 = __fadd_rn(s0, ex2(__fmaf_rn(v[q], sT, -c)));
        }
        float sum = 0.0f;
        if (m > -INFINITY) sum = __fmul_rn(__fadd_rn(s0, s1), ex2(-__fmaf_rn(m, sT, -c)));
        warp_max_sum(m, sum, sT);
        wpart = make_float4(m, sum, 0.0f, 0.0f);
      }
      // leave this warp's partial and count it.  Every warp counts before
      // it releases the stage, and the last warp releases only after it has
      // read the partials, so the next tile in this stage (which needs all
      // eight releases) can reuse neither the count nor the partials early.
      int last = 0;
      if (lane == 0) {
        S.wpart[s][warp] = wpart;
        last = last_warp(S, s);
        if (!last) mbar_arrive(&S.empty[s]);
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        // ---- last warp: combine the eight partials, post the tile ------------
        float2 part;
        float v = -INFINITY, a2 = 0.0f;
        int i = INT_MAX;
        if (lane < kConsumerWarps) {
          const float4 w = S.wpart[s][lane];
          v = w.x;
          a2 = w.y;
          i = __float_as_int(w.y);
        }
        if (tl.greedy) {
          warp_argmax(v, i);
          part = make_float2(v, __int_as_float(i));
        } else {
          warp_max_sum(v, a2, tl.sT);
          part = make_float2(v, a2);
          // the drafted token's logit, if this chunk holds it
          if (lane == 0 && tl.x >= g.e0 && tl.x < g.e0 + g.cnt)
            P.zx[static_cast<size_t>(tl.b) * P.R + tl.r] =
                E::load(buf0 + g.h + (tl.x - g.e0) * E::kBytes);
        }
        __syncwarp();   // every lane has read the partials
        if (lane == 0) {
          mbar_arrive(&S.empty[s]);
          P.part[(static_cast<size_t>(tl.b) * P.R + tl.r) * P.NC + tl.c] = part;
          post_event(S, P, kEvStats, tl.b);
        }
      }
    } else {
      // ---- draw tile: per-warp prefix sums of the final-draw weights ---------
      const unsigned char* rp =
          row_ptr<DT>(P.target, static_cast<size_t>(tl.b) * (K + 1) + tl.t, P.V);
      const Geo gp = chunk_geo<DT>(P, rp, tl.c);
      Geo gq = gp;
      if (tl.residual)
        gq = chunk_geo<DT>(P, row_ptr<DT>(P.draft, static_cast<size_t>(tl.b) * K + tl.t, P.V), tl.c);
      float* out = P.dpart + (static_cast<size_t>(tl.b) * P.NC + tl.c) * 2 * kParts;
      for (int sw = 0; sw < kSweeps; ++sw) {
        const int j = sw * kConsumers + tid;
        float s0 = 0.0f, s1 = 0.0f;
        if (j < gp.nvec) {
          float vp[CH], vq[CH], w0[CH], w1[CH];
          smem_vec<DT>(buf0, gp, j, vp);
          if (tl.residual) {
            if (gq.h == gp.h) {
              smem_vec<DT>(buf1, gq, j, vq);
            } else {
              const int i0 = vec_base<DT>(gp, j);
#pragma unroll
              for (int q = 0; q < CH; ++q) {
                const int i = i0 + q;
                vq[q] = (i >= 0 && i < gp.cnt) ? E::load(buf1 + gq.h + i * E::kBytes) : -INFINITY;
              }
            }
          } else {
#pragma unroll
            for (int q = 0; q < CH; ++q) vq[q] = -INFINITY;
          }
          vec_weights<DT>(vp, vq, tl.residual, tl.Mp, tl.Mq, tl.sT, tl.ratio, w0, w1);
#pragma unroll
          for (int q = 0; q < CH; ++q) {
            s0 = __fadd_rn(s0, w0[q]);
            s1 = __fadd_rn(s1, w1[q]);
          }
        }
        const float i0 = warp_incl_scan(s0, lane);
        const float i1 = warp_incl_scan(s1, lane);
        if (lane == 31) {
          out[sw * kConsumerWarps + warp] = i0;
          out[kParts + sw * kConsumerWarps + warp] = i1;
        }
      }
      if (lane == 31) __threadfence();   // this warp's sums reach L2 before the post
      __syncwarp();
      if (lane == 0) {
        const bool last = last_warp(S, s);   // count first, then release
        mbar_arrive(&S.empty[s]);
        if (last) post_event(S, P, kEvDraw, tl.b);
      }
    }
  }
}

// ---------------------------------------------------------------- control

// Whole warp: (max, sum) of rows [r0, r0 + nr) of request b's partials, row
// r0 + i landing on lane lane0 + i.  The partials are staged into shared
// memory with one lane-parallel sweep of loads, then each lane combines its
// row in chunk order.
__device__ void rows_combine(const Params& P, Ctl& S, const float2* part, int r0, int nr, int lane0,
                             float sT, int lane, float& M, float& Ssum) {
  const int NC = P.NC;
  const int per_round = kCtlBuf / (2 * NC);
  float2* buf = reinterpret_cast<float2*>(S.cbuf);
  for (int g = 0; g < nr; g += per_round) {
    const int cnt = min(per_round, nr - g);
    for (int i = lane; i < cnt * NC; i += 32) buf[i] = __ldcg(part + static_cast<size_t>(r0 + g) * NC + i);
    __syncwarp();
    const int mine = lane - lane0 - g;
    if (mine >= 0 && mine < cnt) {
      M = -INFINITY;
      Ssum = 0.0f;
      for (int c = 0; c < NC; ++c) {
        const float2 p = buf[mine * NC + c];
        pair_combine(M, Ssum, p.x, p.y, sT);
      }
    }
    __syncwarp();
  }
}

// Whole warp: every stats tile of request b is done.  Validates the
// request's tokens and uniforms, combines the partials of every row, runs
// the rule's left-to-right test and either answers the request (greedy) or
// publishes the decision for the owners of the final row's draw tiles.
template <int DT>
__device__ void decide(const Params& P, Ctl& S, int b, int lane) {
  const int K = P.K, R = P.R, NC = P.NC, V = P.V;
  const int n = request_len(P, b);
  const float T = __ldg(P.temperature + b);
  const bool greedy = !(T > 0.0f);
  int tok_bad = 0, u_bad = 0;
  int x_lane = -1;
  float u_lane = 0.0f;
  if (lane < n) {
    x_lane = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + lane);
    tok_bad = (x_lane < 0 || x_lane >= V);
  }
  if (lane <= n) {
    u_lane = __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + lane);
    u_bad = !(u_lane >= 0.0f && u_lane < 1.0f);
  }
  const float ur = __ldg(P.uniforms_resample + b);
  int bad = 0;
  if (__any_sync(0xffffffffu, tok_bad)) bad |= SPECV_DEV_BAD_TOKEN;
  if (__any_sync(0xffffffffu, u_bad) || !(ur >= 0.0f && ur < 1.0f)) bad |= SPECV_DEV_BAD_UNIFORM;
  if (bad) {
    finish_bad(P, b, bad, lane, S.tag);
    return;
  }
  const float2* part = P.part + static_cast<size_t>(b) * R * NC;
  float* rs = P.row_stats ? P.row_stats + static_cast<size_t>(b) * (K + 1) * 8 : nullptr;

  if (greedy) {
    // lane t: argmax of target row t (rows t <= n), chunk partials staged
    float2* buf = reinterpret_cast<float2*>(S.cbuf);
    const int per_round = kCtlBuf / (2 * NC);
    float gv = -INFINITY;
    int g = INT_MAX;
    for (int r0 = 0; r0 <= n; r0 += per_round) {
      const int cnt = min(per_round, n + 1 - r0);
      for (int i = lane; i < cnt * NC; i += 32) buf[i] = __ldcg(part + static_cast<size_t>(r0) * NC + i);
      __syncwarp();
      const int mine = lane - r0;
      if (mine >= 0 && mine < cnt) {
        for (int c = 0; c < NC; ++c) {
          const float2 p = buf[mine * NC + c];
          const int i = __float_as_int(p.y);
          if (better(p.x, i, gv, g)) {
            gv = p.x;
            g = i;
          }
        }
      }
      __syncwarp();
    }
    if (rs && lane <= n) {
      rs[lane * 8 + 0] = gv;
      rs[lane * 8 + 7] = static_cast<float>(g);
    }
    const unsigned miss = __ballot_sync(0xffffffffu, lane < n && g != x_lane);
    const int j = miss ? __ffs(miss) - 1 : n;
    const int gj = __shfl_sync(0xffffffffu, g, j);
    if (gj < 0 || gj >= V) {
      finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, S.tag);
      return;
    }
    if (lane == 0) set_state(P, b, S.tag, kStateNone);   // no draw tiles
    finish_request(P, b, j, gj, lane);
    return;
  }

  // ---- sampled: lane t holds target row t and draft row t ------------------
  const float sT = temp_scale(T);
  float Mp_l = -INFINITY, Sp_l = 0.0f, lp = 0.0f;
  float Mq_l = -INFINITY, Sq_l = 0.0f, lq = 0.0f;
  rows_combine(P, S, part, 0, n + 1, 0, sT, lane, Mp_l, Sp_l);
  rows_combine(P, S, part, K + 1, n, 0, sT, lane, Mq_l, Sq_l);
  if (lane < n) {
    const float zp = __ldcg(P.zx + static_cast<size_t>(b) * R + lane);
    const float zq = __ldcg(P.zx + static_cast<size_t>(b) * R + K + 1 + lane);
    lp = __fsub_rn(__fmul_rn(__fsub_rn(zp, Mp_l), sT), log2f(Sp_l));
    lq = __fsub_rn(__fmul_rn(__fsub_rn(zq, Mq_l), sT), log2f(Sq_l));
  }
  const bool row_bad = (lane <= n && !isfinite(Mp_l)) || (lane < n && !isfinite(Mq_l));
  if (__any_sync(0xffffffffu, row_bad)) {
    finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, S.tag);
    return;
  }
  bool accept = false;
  if (lane < n) accept = __fadd_rn(log2f(u_lane), lq) < lp;
  const unsigned rej = __ballot_sync(0xffffffffu, lane < n && !accept);
  const int j = rej ? __ffs(rej) - 1 : n;
  if (rs) {
    if (lane <= n) {
      rs[lane * 8 + 0] = Mp_l;
      rs[lane * 8 + 1] = Sp_l;
    }
    if (lane < n) {
      rs[lane * 8 + 2] = lp * kLn2;
      rs[lane * 8 + 3] = Mq_l;
      rs[lane * 8 + 4] = Sq_l;
      rs[lane * 8 + 5] = lq * kLn2;
    }
  }
  const float Mp = __shfl_sync(0xffffffffu, Mp_l, j);
  const float Sp = __shfl_sync(0xffffffffu, Sp_l, j);
  const float Mq = __shfl_sync(0xffffffffu, Mq_l, j);
  const float Sq = __shfl_sync(0xffffffffu, Sq_l, j);
  const float u_bonus = __shfl_sync(0xffffffffu, u_lane, n);
  const bool residual = j < n;
  if (lane == 0) {
    Req& q = P.req[b];
    q.j = j;
    q.t_f = j;
    q.residual = residual ? 1 : 0;
    q.u = residual ? ur : u_bonus;
    q.Mp = Mp;
    q.Sp = Sp;
    q.Mq = residual ? Mq : 0.0f;
    q.Sq = residual ? Sq : 1.0f;
    q.sT = sT;
    q.ratio = residual ? __fdiv_rn(Sp, Sq) : 0.0f;
    set_state(P, b, S.tag, kStateDraws);   // release: the fields above first
  }
  __syncwarp();
}

// Whole warp: totals of request b's NC chunks for weight mode `mode` into
// S.ctot (chunk c = sum of its kParts per-warp partials, in order).
__device__ void chunk_totals(const float* dp, int NC, int mode, Ctl& S, int lane) {
  const int per_round = kCtlBuf / kParts;
  for (int c0 = 0; c0 < NC; c0 += per_round) {
    const int cnt = min(per_round, NC - c0);
    for (int i = lane; i < cnt * kParts; i += 32) {
      const int c = i / kParts, k = i - c * kParts;
      S.cbuf[i] = __ldcg(dp + (static_cast<size_t>(c0 + c) * 2 + mode) * kParts + k);
    }
    __syncwarp();
    for (int c = lane; c < cnt; c += 32) {
      float tot = 0.0f;
      for (int k = 0; k < kParts; ++k) tot = __fadd_rn(tot, S.cbuf[c * kParts + k]);
      S.ctot[c0 + c] = tot;
    }
    __syncwarp();
  }
}

// Whole warp: every draw tile of request b is done.  Locates the token from
// the stored prefix sums and one re-read 32-vector segment.
template <int DT>
__device__ void search(const Params& P, Ctl& S, int b, int lane) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec;
  const int K = P.K, NC = P.NC;
  Req q;
  {
    const Req* src = P.req + b;
    q.j = __ldcg(&src->j);
    q.t_f = __ldcg(&src->t_f);
    q.residual = __ldcg(&src->residual);
    q.u = __ldcg(&src->u);
    q.Mp = __ldcg(&src->Mp);
    q.Mq = __ldcg(&src->Mq);
    q.sT = __ldcg(&src->sT);
    q.ratio = __ldcg(&src->ratio);
    q.Sp = __ldcg(&src->Sp);
    q.Sq = __ldcg(&src->Sq);
  }
  const float* dp = P.dpart + static_cast<size_t>(b) * NC * 2 * kParts;
  int mode = 0;
  float W = 0.0f, W_report = 0.0f;
  int owner = -1;
  float tau_c = 0.0f;
  for (int attempt = 0; attempt < 2; ++attempt) {
    chunk_totals(dp, NC, mode, S, lane);
    if (lane == 0) {
      W = 0.0f;
      for (int c = 0; c < NC; ++c) W = __fadd_rn(W, S.ctot[c]);
      const float tau = __fmul_rn(q.u, W);
      float acc = 0.0f, last_acc = 0.0f;
      int last = -1;
      owner = -1;
      for (int c = 0; c < NC; ++c) {
        const float tot = S.ctot[c];
        if (tot > 0.0f) {
          if (owner < 0 && __fadd_rn(acc, tot) > tau) {
            owner = c;
            tau_c = __fsub_rn(tau, acc);
          }
          last = c;
          last_acc = acc;
        }
        acc = __fadd_rn(acc, tot);
      }
      if (owner < 0 && last >= 0) {
        owner = last;
        tau_c = __fsub_rn(tau, last_acc);
      }
    }
    W = __shfl_sync(0xffffffffu, W, 0);
    owner = __shfl_sync(0xffffffffu, owner, 0);
    tau_c = __shfl_sync(0xffffffffu, tau_c, 0);
    __syncwarp();
    if (attempt == 0) W_report = W;
    if (!(q.residual && !(W > 0.0f))) break;
    mode = 1;   // a residual of exactly zero mass: draw from p
  }
  if (owner < 0) {
    finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, S.tag);
    return;
  }
  // the (sweep, warp) segment of the owning chunk
  for (int k = lane; k < kParts; k += 32)
    S.cbuf[k] = __ldcg(dp + (static_cast<size_t>(owner) * 2 + mode) * kParts + k);
  __syncwarp();
  int sel = -1;
  float tau_s = 0.0f;
  if (lane == 0) {
    float acc = 0.0f, last_acc = 0.0f;
    int last = -1;
    for (int k = 0; k < kParts; ++k) {
      const float w = S.cbuf[k];
      if (w > 0.0f) {
        if (sel < 0 && __fadd_rn(acc, w) > tau_c) {
          sel = k;
          tau_s = __fsub_rn(tau_c, acc);
        }
        last = k;
        last_acc = acc;
      }
      acc = __fadd_rn(acc, w);
    }
    if (sel < 0 && last >= 0) {
      sel = last;
      tau_s = __fsub_rn(tau_c, last_acc);
    }
  }
  sel = __shfl_sync(0xffffffffu, sel, 0);
  tau_s = __shfl_sync(0xffffffffu, tau_s, 0);
  __syncwarp();
  if (sel < 0) {
    finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, S.tag);
    return;
  }
  // re-read the segment: lane l holds vector sweep*256 + warp*32 + l
  const bool residual = q.residual && mode == 0;
  const unsigned char* rp = row_ptr<DT>(P.target, static_cast<size_t>(b) * (K + 1) + q.t_f, P.V);
  const unsigned char* rq =
      q.residual ? row_ptr<DT>(P.draft, static_cast<size_t>(b) * K + q.t_f, P.V) : nullptr;
  const Geo gp = chunk_geo<DT>(P, rp, owner);
  const int j = (sel / kConsumerWarps) * kConsumers + (sel % kConsumerWarps) * 32 + lane;
  float vp[CH], vq[CH], w0[CH], w1[CH];
  const int i0 = vec_base<DT>(gp, j);
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int i = i0 + k;
    const bool in = j < gp.nvec && i >= 0 && i < gp.cnt;
    vp[k] = in ? E::ldg(rp + static_cast<size_t>(gp.e0 + i) * E::kBytes) : -INFINITY;
    vq[k] = (in && residual) ? E::ldg(rq + static_cast<size_t>(gp.e0 + i) * E::kBytes) : -INFINITY;
  }
  vec_weights<DT>(vp, vq, residual, q.Mp, q.Mq, q.sT, q.ratio, w0, w1);
  float* w = mode == 0 ? w0 : w1;
  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    if (!(vp[k] > -INFINITY)) w[k] = 0.0f;   // outside the chunk
    sum = __fadd_rn(sum, w[k]);
  }
  const float incl = warp_incl_scan(sum, lane);
  const unsigned hit = __ballot_sync(0xffffffffu, sum > 0.0f && incl > tau_s);
  const unsigned pos = __ballot_sync(0xffffffffu, sum > 0.0f);
  const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  if (l < 0) {
    finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, S.tag);
    return;
  }
  const float excl = __shfl_sync(0xffffffffu, incl - sum, l);
  int tok = -1;
  if (lane == l) {
    const float tau3 = __fsub_rn(tau_s, excl);
    float run = 0.0f;
    int pick = -1, lastq = -1;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      if (w[k] > 0.0f) {
        run = __fadd_rn(run, w[k]);
        if (pick < 0 && run > tau3) pick = k;
        lastq = k;
      }
    }
    if (pick < 0) pick = lastq;
    tok = gp.e0 + i0 + pick;
  }
  tok = __shfl_sync(0xffffffffu, tok, l);
  if (P.row_stats && lane == 0) {
    float* rs = P.row_stats + (static_cast<size_t>(b) * (K + 1) + q.t_f) * 8;
    rs[6] = __fdiv_rn(W_report, q.Sp);
    rs[7] = static_cast<float>(tok);
  }
  if (tok < 0 || tok >= P.V) {
    finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, S.tag);
    return;
  }
  finish_request(P, b, q.j, tok, lane);
}

// The control warp: takes the consumers' events in runs (every event that is
// already posted), adds each run's tiles to the request counters with one
// atomic per request, and runs the decision or the search for a request
// whose last tile it counted.
template <int DT>
__device__ void control(const Params& P, Ctl& S, int lane) {
  int e = 0;
  bool stop = false;
  while (!stop) {
    const int slot0 = e % kMailbox;
    const uint32_t ph0 = static_cast<uint32_t>(e / kMailbox) & 1u;
    if (!warp_wait(&S.mb_full[slot0], ph0, lane)) {
      if (lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
      return;
    }
    // gather the run (lane 0), release the mailbox slots
    int runs = 0;
    if (lane == 0) {
      for (;;) {
        const int slot = e % kMailbox;
        const uint32_t ph = static_cast<uint32_t>(e / kMailbox) & 1u;
        if (!mbar_test(&S.mb_full[slot], ph)) break;   // nothing more posted yet
        const int2 evt = S.mb[slot];
        mbar_arrive(&S.mb_empty[slot]);
        ++e;
        if (evt.x == kEvSentinel) {
          stop = true;
          break;
        }
        if (runs > 0 && S.run_kind[runs - 1] == evt.x && S.run_b[runs - 1] == evt.y) {
          ++S.run_cnt[runs - 1];
        } else {
          S.run_kind[runs] = evt.x;
          S.run_b[runs] = evt.y;
          S.run_cnt[runs] = 1;
          ++runs;
          if (runs == kRunMax) break;
        }
      }
    }
    runs = __shfl_sync(0xffffffffu, runs, 0);
    stop = __shfl_sync(0xffffffffu, stop, 0);
    e = __shfl_sync(0xffffffffu, e, 0);
    __syncwarp();
    // one atomic per run, the runs' atomics in flight together on their lanes
    int last = 0;
    if (lane < runs) {
      const int kind = S.run_kind[lane], b = S.run_b[lane], cnt = S.run_cnt[lane];
      if (kind == kEvStats) {
        const int n = request_len(P, b);
        const float T = __ldg(P.temperature + b);
        const int prev = AtomicInt(P.req[b].stats_done).fetch_add(cnt, cuda::memory_order_acq_rel);
        last = prev + cnt == request_tiles(P, n, T);
      } else {
        const int prev = AtomicInt(P.req[b].draw_done).fetch_add(cnt, cuda::memory_order_acq_rel);
        last = prev + cnt == P.NC;
      }
    }
    const unsigned lasts = __ballot_sync(0xffffffffu, last);
    __syncwarp();   // every lane reads after the acquiring lanes
    for (int i = 0; i < runs; ++i) {
      if (!((lasts >> i) & 1u)) continue;
      const int kind = S.run_kind[i], b = S.run_b[i];
      if (kind == kEvStats) decide<DT>(P, S, b, lane);
      else search<DT>(P, S, b, lane);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- kernel

template <int DT>
__global__ void __launch_bounds__(kThreads) verify_kernel(const Params P) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  __shared__ Ctl S;
  extern __shared__ __align__(128) unsigned char dyn[];

  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);   // each consumer warp releases
      S.done_cnt[s] = 0;
    }
    S.mb_head = 0;
    for (int i = 0; i < kMailbox; ++i) {
      mbar_init(&S.mb_full[i], 1);
      mbar_init(&S.mb_empty[i], 1);
    }
    S.tag = (static_cast<uint32_t>(P.header[kHEpoch]) + 1u) & 0x3FFFFFFFu;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == kProducerWarp)
    producer<DT>(P, S, dyn, tid & 31);
  else if (warp == kControlWarp)
    control<DT>(P, S, tid & 31);
  else
    consumer<DT>(P, S, dyn, tid);

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(P.header + kHExit, 1);
    if (prev == static_cast<int>(gridDim.x) - 1) {
      // last CTA of the launch: every ticket is taken and every request
      // answered; reset for the next call
      P.header[kHExit] = 0;
      P.header[kHEpoch] = P.header[kHEpoch] + 1;
    }
  }
}

// ---------------------------------------------------------------- host side

int elt_bytes(specv_dtype dt) { return dt == SPECV_BF16 ? 2 : 4; }

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (!v || !*v) return fallback;
  const int x = std::atoi(v);
  return x > 0 ? x : fallback;
}

struct Layout {
  size_t header, req, part, zx, dpart, total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

Layout ws_layout(int B, int K, int NC) {
  const size_t R = 2 * static_cast<size_t>(K) + 1;
  Layout L;
  L.header = 0;
  L.req = kHeaderBytes;
  L.part = align256(L.req + sizeof(Req) * static_cast<size_t>(B));
  L.zx = align256(L.part + sizeof(float2) * B * R * NC);
  L.dpart = align256(L.zx + sizeof(float) * B * R);
  L.total = align256(L.dpart + sizeof(float) * static_cast<size_t>(B) * NC * 2 * kParts);
  return L;
}

int chunks_per_row(int V, specv_dtype dt) {
  const int ce = kChunkBytes / elt_bytes(dt);
  return (V + ce - 1) / ce;
}

int stage_count() {
  int s = env_int("SPECV_STAGES", 3);
  if (s < 1) s = 1;
  if (s > kMaxStages) s = kMaxStages;
  return s;
}

// Resident CTAs per SM for a stage count, cached per device.
template <int DT>
cudaError_t resident_ctas(int stages, int* out) {
  static std::mutex mu;
  static int cache[64][kMaxStages + 1];
  static bool attr_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxStages * kStageBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (!cache[dev][stages]) {
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<DT>, kThreads,
                                                      static_cast<size_t>(stages) * kStageBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cache[dev][stages] = per_sm * sms;
  }
  *out = cache[dev][stages];
  return cudaSuccess;
}

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
      !aligned(out_tokens, 4) || !aligned(workspace, 256) || (row_stats && !aligned(row_stats, 4)))
    return SPECV_ERR_INVALID_ARG;
  if (workspace_bytes < specv_workspace_bytes(B, K, V, dtype)) return SPECV_ERR_WORKSPACE;

  const int NC = chunks_per_row(V, dtype);
  const int stages = stage_count();
  int ctas = 0;
  cudaError_t e = dtype == SPECV_BF16 ? resident_ctas<SPECV_BF16>(stages, &ctas)
                                      : resident_ctas<SPECV_F32>(stages, &ctas);
  if (e != cudaSuccess || ctas < 1) return SPECV_ERR_CUDA;
  const long long groups = static_cast<long long>(B) * (2 * K + 1) * ((NC + kGroup - 1) / kGroup);
  const int grid = static_cast<int>(groups < ctas ? groups : ctas);

  const Layout L = ws_layout(B, K, NC);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
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
  P.R = 2 * K + 1;
  P.NC = NC;
  P.NG = (NC + kGroup - 1) / kGroup;
  P.CE = kChunkBytes / static_cast<int>(eb);
  P.stages = stages;
  P.accepted_len = accepted_len;
  P.out_tokens = out_tokens;
  P.header = reinterpret_cast<int32_t*>(ws + L.header);
  P.req = reinterpret_cast<Req*>(ws + L.req);
  P.part = reinterpret_cast<float2*>(ws + L.part);
  P.zx = reinterpret_cast<float*>(ws + L.zx);
  P.dpart = reinterpret_cast<float*>(ws + L.dpart);
  P.row_stats = row_stats;

  const size_t smem = static_cast<size_t>(stages) * kStageBytes;
  if (dtype == SPECV_BF16)
    verify_kernel<SPECV_BF16><<<grid, kThreads, smem, stream>>>(P);
  else
    verify_kernel<SPECV_F32><<<grid, kThreads, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? SPECV_OK : SPECV_ERR_CUDA;
}

size_t pad256(size_t x) { return align256(x); }

// ---------------------------------------------------------------- no-allocation scratch
//
// Scratch for spec_verify_sample_noalloc: the same layout as a caller's
// workspace, at most SPECV_NOALLOC_SCRATCH_BYTES.  It is a module-scope
// device array, so every GPU that loads this library holds it until the
// process exits, and every call on a device shares it.
__device__ __align__(256) unsigned char g_noalloc_scratch[SPECV_NOALLOC_SCRATCH_BYTES];

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

int specv_version(void) { return 300; }

int specv_max_vocab(specv_dtype dtype) {
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return 0;
  return kMaxChunks * (kChunkBytes / elt_bytes(dtype));
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

size_t specv_workspace_bytes(int B, int K, int V, specv_dtype dtype) {
  if (B < 1 || K < 1 || V < 1 || B > SPECV_MAX_BATCH || K > SPECV_MAX_DRAFT ||
      (dtype != SPECV_F32 && dtype != SPECV_BF16) || V > specv_max_vocab(dtype))
    return 0;
  return ws_layout(B, K, chunks_per_row(V, dtype)).total;
}

specv_status specv_workspace_init(void* workspace, size_t workspace_bytes, specv_stream_t stream) {
  if (!workspace || !aligned(workspace, 256) || workspace_bytes == 0) return SPECV_ERR_INVALID_ARG;
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
  if (!workspace || !status || workspace_bytes < static_cast<size_t>(kHeaderBytes))
    return SPECV_ERR_INVALID_ARG;
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
  (void)with_draft;
  if (!out || specv_workspace_bytes(B, K, V, dtype) == 0) return SPECV_ERR_INVALID_ARG;
  const int stages = stage_count();
  int ctas = 0;
  const cudaError_t e = dtype == SPECV_BF16 ? resident_ctas<SPECV_BF16>(stages, &ctas)
                                            : resident_ctas<SPECV_F32>(stages, &ctas);
  if (e != cudaSuccess) return SPECV_ERR_CUDA;
  const int NC = chunks_per_row(V, dtype);
  const long long groups = static_cast<long long>(B) * (2 * K + 1) * ((NC + kGroup - 1) / kGroup);
  out[0] = static_cast<int32_t>(groups < ctas ? groups : ctas);
  out[1] = kChunkBytes / elt_bytes(dtype);
  out[2] = stages;
  out[3] = NC;
  out[4] = stages * kStageBytes;
  out[5] = kThreads;
  return SPECV_OK;
}

specv_status spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                        specv_dtype dtype, const int32_t* draft_tokens,
                                        const int32_t* draft_len, const float* temperature,
                                        const float* uniforms, const float* uniforms_resample,
                                        int B, int K, int V, int32_t* accepted_len,
                                        int32_t* out_tokens, specv_stream_t stream) {
  const size_t bytes = specv_workspace_bytes(B, K, V, dtype);
  if (bytes == 0) return SPECV_ERR_INVALID_ARG;
  if (bytes > SPECV_NOALLOC_SCRATCH_BYTES) return SPECV_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return SPECV_ERR_CUDA;
  // The array keeps the previous call's contents: zero the part this call uses.
  if (cudaMemsetAsync(scratch, 0, bytes, s) != cudaSuccess) return SPECV_ERR_CUDA;
  return launch(target_logits, draft_logits, dtype, draft_tokens, draft_len, temperature, uniforms,
                uniforms_resample, B, K, V, accepted_len, out_tokens, scratch, bytes, nullptr, s);
}

}  // extern "C"
