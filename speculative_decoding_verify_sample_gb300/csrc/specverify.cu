// libspecverify: the speculative-decoding verification sampler for GB300
// (sm_103a), as a short chain of kernels on the caller's stream.
//
// The rule ("Decodificación Especulativa y EAGLE", Phase 10 - Lesson 25,
// sections "El Concepto", "La Regla de Exactitud", "Caso codicioso"): for
// each request, accept drafted tokens left to right while u_t < p(x_t)/q(x_t);
// at the first rejection draw a replacement from (p - q)+ and stop; if every
// draft is accepted draw a bonus token from p at the next position; at
// temperature 0 compare argmax(p) with the draft instead.
//
// Design: up to four kernels on the caller's stream, each launched as a
// programmatic dependent so its launch and prologue overlap the previous
// kernel's tail; each waits for the previous kernel before it writes.
//
//  1. stats_kernel streams every row a request needs (target rows t <= n,
//     draft rows t < n when sampled) once from HBM with TMA bulk copies,
//     in 6 KB chunks: first every row but the position-0 pairs, then those
//     pairs, so that the pairs a rejection most often re-reads are the ones
//     left in L2.  Each warp is an agent with a private ring of kSlots
//     shared-memory slots (32 warps with one slot each: the other warps'
//     copies and reductions hide each one's wait); warp g of the grid's G
//     takes chunks g, g + G, g + 2 G, ... (decoded 32 at a time, one per
//     lane).  A chunk is reduced to a record: its maximum and sum of
//     exp((z - max)/T), or at T = 0 its maximum and lowest argmax.  The
//     chunk holding a drafted token also records that token's logit.  The
//     copies stream with an L2 evict-first policy, the records are stored
//     evict-last.
//  2. decide_kernel, one CTA per request, combines the records, runs the
//     left-to-right accept test (or the greedy comparison) and writes the
//     outputs.  A request whose drafts are all accepted gets its bonus
//     draw's chunk here (from row n's records) and joins a bonus list; a
//     rejected sampled request joins the residual list.  The sampler and
//     the one-hot rule make their walks here instead and stop after this
//     kernel; greedy trees too.
//  3. residual_kernel reads the rejected rows again (target and draft, in
//     3 KB pieces) and sums (p - q)+ per piece and per 512-byte sweep.
//     Warps of its own take the bonus draws meanwhile: the listed chunk
//     read once more, its sweeps summed four at a time to the token.
//  4. search_kernel, one warp per listed request, draws its token: the
//     piece from the piece sums, the sweep from that piece's sweep sums,
//     the token from the sweep of both rows read again.
//
// Beside them: insert_kernel (the post-accept insert, one CTA) and
// gather_rows_kernel (the host entry point's copy of the needed rows of
// page-locked logits over the host link).
//
// The only waits are a warp's waits on its own bulk copies; each is
// bounded in time and sets a status bit when it gives up.  No warp waits on
// data another warp or CTA produces: kernel boundaries order all of it.

#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "specverify.h"

namespace {

constexpr int kAgents = 32;                             // agent warps per CTA
constexpr int kThreads = kAgents * 32;
constexpr int kSlots = 1;                               // ring slots per agent
constexpr int kChunkBytes = 6144;                       // deciding / bonus item: one chunk of one row
constexpr int kDrawBytes = 3072;                        // residual piece: this much of each row
constexpr int kDrawSweeps = kDrawBytes / 512;           // 32 lanes x 16 bytes per sweep
constexpr int kDraftOff = kDrawBytes;                   // draft part of a residual slot
constexpr int kPieceRec = 8;                            // floats per piece record: sweep sums, total, unused
static_assert(kDrawSweeps + 1 <= kPieceRec && kPieceRec % 4 == 0, "a piece record is whole 16-byte words");
constexpr int kSlotBytes = kChunkBytes + 32;
constexpr int kRingBytes = kAgents * kSlots * kSlotBytes;
constexpr int kPlanMax = 1024;                          // requests per launch (the host splits)
constexpr int kDecideWarps = 4;                         // warps of a decide / search CTA
constexpr int kMaxRowBytes = 1 << 21;                   // 2 MB per row of logits
constexpr int kMaxChunks = (kMaxRowBytes + 15 + kChunkBytes - 1) / kChunkBytes;
constexpr int kMaxDrawChunks = (kMaxRowBytes + 15 + kDrawBytes - 1) / kDrawBytes;
constexpr long long kWaitLimitCycles = 4000000000ll;    // ~2 s at 2 GHz
constexpr uint32_t kSuspendHintNs = 20000;

static_assert(kSlotBytes >= kDraftOff + kDrawBytes + 16, "residual slot too small");
static_assert(kSlotBytes % 16 == 0, "slots must keep 16-byte alignment");
static_assert(kMaxChunks * 8 <= kSlotBytes, "the records of one row fit a slot");
static_assert(kMaxDrawChunks * 4 <= kSlotBytes, "the residual masses of one row fit a slot");
static_assert(kMaxChunks < 512, "a stats chunk index fits 9 bits");
static_assert(kPlanMax <= 1024 && 2 * SPECV_MAX_DRAFT + 1 < 64, "a request fits 10 bits, a row 6");

// workspace header words (int32 index), one 128-byte line each: the device
// status, and the lengths of the residual and bonus lists (the stats kernel
// empties both lists at the start of every launch sequence)
constexpr int kHStatus = 0, kHResid = 96, kHBonus = 160;
constexpr int kHeaderBytes = 1024;
static_assert((kHBonus + 1) * 4 <= kHeaderBytes, "header words fit the header");



constexpr int kItemA = 1, kItemR = 3;

// What a launch sequence computes (Params::mode).
constexpr int kModeVerify = 0;   // the verification rule, draft logits given
constexpr int kModeSample = 1;   // the draft-side sampler: one row per request, no drafts
constexpr int kModeOnehot = 2;   // the rule for a draft that proposes its top token (q one-hot)
constexpr int kModeTree = 3;     // greedy verification of a token tree (rows = tree nodes)
constexpr int kMaxTreeNodes = 64;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A listed draw (32 bytes), written by the decision: entry e of the
// residual list (e counted up from 0) or of the bonus list (counted down
// from B - 1), so the draw's kernel reads everything it needs at once.
struct __align__(16) Req {
  int b;          // the request
  int j;          // the rejected row (a bonus draw: n)
  float aux;      // residual: S_p of the rejected row; bonus: the target mass left at its chunk
  int chunk;      // bonus: its chunk of row n; residual: uniforms_resample[b] (float bits)
  float4 prm;     // Mp, Mq, log2(e)/T, S_p/S_q of the rejected row (a bonus draw: Mp, 0, log2(e)/T, 0)
};
static_assert(sizeof(Req) == 32, "Req is one 32-byte record");

struct Params {
  const unsigned char* target;
  const unsigned char* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  const float* uniforms;
  const float* uniforms_resample;
  int B, K, V;
  int mode;         // kModeVerify / kModeSample / kModeOnehot / kModeTree
  const int32_t* parents;   // tree mode: [B][K+1] parent of each node (-1 at the root)
  int32_t* path_nodes;      // tree mode: [B][K+1] the accepted path's nodes
  int R;            // record rows per request: K+1 target, then K draft
  int NC;           // stats chunks per row
  int NCd;          // residual pieces per row
  float inv_NC;     // 1 / NC
  // 16-byte-aligned address ranges the bulk copies may read
  uintptr_t t_lo, t_hi, d_lo, d_hi;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t* header;
  Req* req;         // [B] listed draws (counts: header[kHResid], header[kHBonus])
  uint2* part;      // [B][R][NC] chunk records: (max, sum) or (max, index)
  float* zx;        // [B][R] the drafted token's logit in rows t < n
  float* dpc;       // [B][NCd][kPieceRec] residual sums of each piece: its sweeps, then its total (by list entry)
  float* row_stats; // [B][K+1][8] or null
};

// The call's plan, built by every CTA of the stats kernel: the rows each
// request needs (prefix sums) and its length.  The stream takes the rows in
// two passes: first every row but the position-0 pairs (target row 0 and
// draft row 0 of a request with draft rows), then those pairs.  Position 0
// is where a rejection is likeliest, and the pairs read last are the ones
// still in L2 when the residual pass reads a rejected pair again.
struct Plan {
  int rb[kPlanMax + 1];       // first-pass rows before request b
  int rb2[kPlanMax + 1];      // second-pass rows (0 or 2 per request) before request b
  uint8_t info[kPlanMax];     // draft length | 0x40 | 0x80 if the request samples (0: unusable)
  int total1;                 // tickets of the first pass
  int total;                  // tickets: chunks of every needed row
};

// One item as its agent staged it.
struct __align__(16) Item {
  int kind;     // kItemA (a stats chunk) / kItemR (a residual piece pair)
  int b;
  int row;      // record row: t (target) or K+1+t (draft); residual: the rejected t
  int c;        // chunk
  int n;        // the request's draft length
  float sT;     // log2(e)/T (0: greedy)
  int x;        // drafted token of the row (rows t < n of sampled requests), else -1
  float4 prm;   // residual: the decision's Mp, Mq, log2(e)/T, S_p/S_q
};

struct AgentSmem {
  uint64_t bar[kSlots];
  Item item[kSlots];   // the items in the slots
};

struct Smem {
  Plan plan;
  AgentSmem ag[kAgents];
  int red[kAgents * 2];
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
    __device__ float value() const { return vec_max(make_uint4(w[0], w[1], w[2], w[3])); }
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

// Whole warp: waits for phase `parity` of the barrier; gives up after
// kWaitLimitCycles.  Every lane polls, so every lane acquires the phase.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  bool ok = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, ok)) return true;
  const long long t0 = clock64();
  for (;;) {
    ok = ok || mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if (__any_sync(0xffffffffu, clock64() - t0 > kWaitLimitCycles)) return false;
  }
}

// Orders this thread's earlier shared-memory accesses (generic proxy) before
// later bulk copies into the same bytes (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 cache policies: lines of the logits are streamed once (or read once
// more soon after) and leave L2 first, so the small state the later kernels
// read (chunk records, the lists, the per-request inputs) stays resident.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Non-tensor TMA bulk copy global -> this CTA's shared memory, with L2
// policy `pol`.  Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, uintptr_t src, uint32_t bytes,
                                              uint64_t* bar, uint64_t pol) {
  const unsigned long long gsrc =
      static_cast<unsigned long long>(__cvta_generic_to_global(reinterpret_cast<const void*>(src)));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// An 8-byte store that L2 keeps in preference to streamed lines.
__device__ __forceinline__ void st_keep(uint2* p, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x), "r"(v.y),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// 2^x on the MUFU unit (PTX ex2.approx.ftz.f32); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp((z - m)/T) as 2^((z - m) * log2(e)/T), the argument formed from the
// difference to the reference m.
__device__ __forceinline__ float scaled_exp(float z, float m, float sT) {
  return ex2(__fmul_rn(__fsub_rn(z, m), sT));
}

// Pairs of fp32 values in one 64-bit register pair, for the two-wide FP32
// instructions of the sm_100 family (add / sub / mul / fma .rn.f32x2).
// Each half is rounded exactly as the scalar instruction rounds it, so a
// paired computation gives the scalar one's bits.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void up2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ float temp_scale(float T) { return __fdiv_rn(kLog2e, T); }

// ---------------------------------------------------------------- reductions

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

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = __fadd_rn(v, y);
  }
  return v;
}

__device__ __forceinline__ int warp_incl_scan_int(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// ---------------------------------------------------------------- geometry

// A chunk of a row as it sits in a slot.  Slot byte 0 is global address g0;
// the row's element e is at slot byte off0 + e * elt; elements [e_lo, e_hi)
// belong to the chunk.  For the target row of any item g0 is the 16-byte
// boundary at or below the row's start plus c * CB, so the slot's 16-byte
// vectors are the row's aligned vectors.
struct Chunk {
  uintptr_t g0;
  int off0;
  int e_lo, e_hi;
};

template <int DT>
__device__ __forceinline__ uintptr_t row_addr(const unsigned char* base, size_t row, int V) {
  return reinterpret_cast<uintptr_t>(base) + row * static_cast<size_t>(V) * Elt<DT>::kBytes;
}

template <int DT>
__device__ __forceinline__ Chunk chunk_of(uintptr_t row, int V, int c, int CB) {
  constexpr int eb = Elt<DT>::kBytes;
  const uintptr_t a0 = row & ~static_cast<uintptr_t>(15);
  const int h = static_cast<int>(row - a0);   // a multiple of the element size
  Chunk k;
  k.g0 = a0 + static_cast<size_t>(c) * CB;
  k.off0 = h - c * CB;
  k.e_lo = max(0, (c * CB - h) / eb);
  k.e_hi = min(V, ((c + 1) * CB - h) / eb);
  return k;
}

// The draft elements [e_lo, e_hi) of a draw chunk, placed from the 16-byte
// boundary at or below the first of them.
template <int DT>
__device__ __forceinline__ Chunk draft_part(uintptr_t row, const Chunk& tgt) {
  constexpr int eb = Elt<DT>::kBytes;
  Chunk k;
  const uintptr_t first = row + static_cast<size_t>(max(tgt.e_lo, 0)) * eb;
  k.g0 = first & ~static_cast<uintptr_t>(15);
  k.off0 = static_cast<int>(static_cast<intptr_t>(row) - static_cast<intptr_t>(k.g0));
  k.e_lo = tgt.e_lo;
  k.e_hi = tgt.e_hi;
  return k;
}

// The bytes of a chunk a bulk copy moves: the 16-byte-aligned cover of its
// elements, inside the tensor's aligned range [lo, hi).  Returns the byte
// count (0: nothing) and the global start.
template <int DT>
__device__ __forceinline__ uint32_t bulk_span(const Chunk& k, uintptr_t lo, uintptr_t hi,
                                              uintptr_t* start) {
  constexpr int eb = Elt<DT>::kBytes;
  if (k.e_hi <= k.e_lo) return 0;
  const uintptr_t first = k.g0 + static_cast<intptr_t>(k.off0) + static_cast<intptr_t>(k.e_lo) * eb;
  const uintptr_t end = k.g0 + static_cast<intptr_t>(k.off0) + static_cast<intptr_t>(k.e_hi) * eb;
  const uintptr_t a = first & ~static_cast<uintptr_t>(15);
  const uintptr_t z = (end + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t s = a > lo ? a : lo;
  const uintptr_t e = z < hi ? z : hi;
  if (e <= s) return 0;
  *start = s;
  return static_cast<uint32_t>(e - s);
}

// Whole warp: elements of the chunk that lie outside the tensor's aligned
// range (at most 15 bytes at either end of a tensor) are loaded by lanes.
template <int DT>
__device__ __noinline__ void fix_edges_slow(const Chunk& k, uintptr_t g_first, uintptr_t g_end,
                                            uintptr_t lo, uintptr_t hi, unsigned char* slot,
                                            int lane);

template <int DT>
__device__ __forceinline__ void fix_edges(const Chunk& k, uintptr_t lo, uintptr_t hi,
                                          unsigned char* slot, int lane) {
  constexpr int eb = Elt<DT>::kBytes;
  if (k.e_hi <= k.e_lo) return;
  const uintptr_t g_first = k.g0 + static_cast<intptr_t>(k.off0) + static_cast<intptr_t>(k.e_lo) * eb;
  const uintptr_t g_end = k.g0 + static_cast<intptr_t>(k.off0) + static_cast<intptr_t>(k.e_hi) * eb;
  if (g_first >= lo && g_end <= hi) return;   // the common case: nothing outside
  fix_edges_slow<DT>(k, g_first, g_end, lo, hi, slot, lane);
}

template <int DT>
__device__ __noinline__ void fix_edges_slow(const Chunk& k, uintptr_t g_first, uintptr_t g_end,
                                            uintptr_t lo, uintptr_t hi, unsigned char* slot,
                                            int lane) {
  constexpr int eb = Elt<DT>::kBytes;
  const uintptr_t h1 = g_end < lo ? g_end : lo;                 // head [g_first, h1)
  uintptr_t t0 = g_first > hi ? g_first : hi;                   // tail [t0, g_end)
  if (t0 < h1) t0 = h1;
  const int nh = h1 > g_first ? static_cast<int>((h1 - g_first) / eb) : 0;
  const int nt = g_end > t0 ? static_cast<int>((g_end - t0) / eb) : 0;
  if (nh == 0 && nt == 0) return;
  if (lane < nh) {
    const uintptr_t g = g_first + static_cast<uintptr_t>(lane) * eb;
    Elt<DT>::copy1(slot + (g - k.g0), reinterpret_cast<const unsigned char*>(g));
  } else if (lane >= 16 && lane - 16 < nt) {
    const uintptr_t g = t0 + static_cast<uintptr_t>(lane - 16) * eb;
    Elt<DT>::copy1(slot + (g - k.g0), reinterpret_cast<const unsigned char*>(g));
  }
  __syncwarp();
}

// Vectors of a target chunk: fully valid vectors [vf0, vf1), and up to two
// partly valid edge vectors va (first) and vb (last) (-1: none).
struct Vecs {
  int e_base;      // element of vector 0, part 0 (may be negative)
  int vf0, vf1;
  int va, vb;
};

template <int DT>
__device__ __forceinline__ Vecs vecs_of(const Chunk& k) {
  constexpr int CH = Elt<DT>::kPerVec, eb = Elt<DT>::kBytes;
  Vecs v;
  v.e_base = -k.off0 / eb;
  v.va = v.vb = -1;
  if (k.e_hi <= k.e_lo) {
    v.vf0 = v.vf1 = 0;
    return v;
  }
  const int lo = k.e_lo - v.e_base, hi = k.e_hi - v.e_base;   // element offsets in the slot
  v.vf0 = (lo + CH - 1) / CH;
  v.vf1 = hi / CH;
  if (lo % CH) v.va = lo / CH;
  if (hi % CH) v.vb = hi / CH;
  if (v.vf1 < v.vf0) {   // the whole chunk inside one vector
    v.vf1 = v.vf0;
    v.va = lo / CH;
    v.vb = -1;
  } else if (v.va >= 0 && v.va == v.vb) {
    v.vb = -1;
  }
  return v;
}

// Values of vector j with elements outside [e_lo, e_hi) set to -inf.
template <int DT>
__device__ __forceinline__ void masked_vec(const unsigned char* slot, const Vecs& vs,
                                           const Chunk& k, int j, float* v) {
  using E = Elt<DT>;
  E::unpack(reinterpret_cast<const uint4*>(slot)[j], v);
  const int e0 = vs.e_base + j * E::kPerVec;
#pragma unroll
  for (int q = 0; q < E::kPerVec; ++q)
    if (e0 + q < k.e_lo || e0 + q >= k.e_hi) v[q] = -INFINITY;
}

// ---------------------------------------------------------------- requests

// A request's draft length n: its drafted tokens, or (sampler) 0, or (tree)
// its node count less the root.
__device__ __forceinline__ int request_len(const Params& P, int b) {
  if (P.mode == kModeTree) return __ldg(P.draft_len + b) - 1;
  return P.draft_len ? __ldg(P.draft_len + b) : P.K;
}

__device__ __forceinline__ float request_T(const Params& P, int b) {
  return P.temperature ? __ldg(P.temperature + b) : 0.0f;
}

__device__ __forceinline__ int request_bad(const Params& P, int n, float T) {
  const int lo = (P.mode == kModeSample || P.mode == kModeTree) ? 0 : 1;
  if (n < lo || n > P.K) return SPECV_DEV_BAD_DRAFT_LEN;
  if (!(T >= 0.0f) || isinf(T)) return SPECV_DEV_BAD_TEMPERATURE;
  if (T > 0.0f && P.draft == nullptr && P.mode == kModeVerify) return SPECV_DEV_NO_DRAFT;
  return 0;
}

// Whether a request's rows include draft rows: a sampled request of the
// verification rule (a one-hot draft has no logits; the sampler and trees
// have no drafts).
__device__ __forceinline__ bool two_rows(const Params& P, bool sampled) {
  return sampled && P.mode == kModeVerify;
}

// Rows a usable request needs: target rows t <= n, and draft rows t < n
// when it samples with draft logits.
__device__ __forceinline__ int request_rows(const Params& P, int n, float T) {
  return two_rows(P, T > 0.0f) ? 2 * n + 1 : n + 1;
}

// Record row of a request's row slot: a request with draft rows alternates
// target row t and draft row t in its first 2n slots, slot 2n is target row
// n; otherwise its slots are its target rows.
__device__ __forceinline__ int slot_row(int slot, bool both, int n, int K) {
  if (!both || slot == 2 * n) return both ? n : slot;
  return (slot & 1) ? K + 1 + (slot >> 1) : (slot >> 1);
}

// Whole warp: out_tokens[b] = x_0 .. x_{j-1}, tok at j, -1 after;
// accepted_len[b] = j (j = -1: every entry -1).  Lane s < j holds x_s.
__device__ __forceinline__ void write_outputs(const Params& P, int b, int j, int tok, int x_lane,
                                              int lane) {
  for (int s = lane; s <= P.K; s += 32)
    P.out_tokens[static_cast<size_t>(b) * (P.K + 1) + s] =
        j < 0 ? -1 : (s < j ? x_lane : (s == j ? tok : -1));
  if (lane == 0 && P.accepted_len) P.accepted_len[b] = j;
}

// ---------------------------------------------------------------- plan

// A usable request's rows in the two passes, packed (second << 16) | first:
// a request with draft rows reads its position-0 pair in the second pass.
__device__ __forceinline__ int plan_rows(const Params& P, int n, float T) {
  const int all = request_rows(P, n, T);
  return two_rows(P, T > 0.0f) ? ((2 << 16) | (all - 2)) : all;
}

// Whole CTA: builds the call's plan: the rows each request needs, as
// prefix sums.  A request whose length or temperature is unusable needs no
// rows (the decision kernel answers it).
__device__ void build_plan(const Params& P, Plan& pl, int* red) {
  const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, w = tid >> 5;
  const int B = P.B;
  const int per = (B + kThreads - 1) / kThreads;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  // rows of the two passes packed as (second << 16) | first: a request has
  // at most 2 K + 1 <= 33 rows, so the first-pass sum stays below 2^16
  int rows = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = request_len(P, b);
    const float T = request_T(P, b);
    if (!request_bad(P, n, T)) rows += plan_rows(P, n, T);
  }
  const int ir = warp_incl_scan_int(rows, lane);
  if (lane == 31) red[w] = ir;
  __syncthreads();
  int r = ir - rows, tr = 0;
#pragma unroll
  for (int k = 0; k < kAgents; ++k) {
    if (k < w) r += red[k];
    tr += red[k];
  }
  for (int b = b0; b < b1; ++b) {
    const int n = request_len(P, b);
    const float T = request_T(P, b);
    const bool bad = request_bad(P, n, T) != 0;
    pl.rb[b] = r & 0xFFFF;
    pl.rb2[b] = r >> 16;
    pl.info[b] = static_cast<uint8_t>(bad ? 0 : (n | 0x40 | (T > 0.0f ? 0x80 : 0)));
    if (!bad) r += plan_rows(P, n, T);
  }
  if (tid == 0) {
    pl.rb[B] = tr & 0xFFFF;
    pl.rb2[B] = tr >> 16;
    pl.total1 = (tr & 0xFFFF) * P.NC;
    pl.total = ((tr & 0xFFFF) + (tr >> 16)) * P.NC;
  }
  __syncthreads();
}

// m / NC for 0 <= m < 2^24: a float estimate (exact operands) corrected by
// one either way.
__device__ __forceinline__ int div_nc(const Params& P, int m) {
  int r = __float2int_rz(__int2float_rn(m) * P.inv_NC);
  if (r * P.NC > m) --r;
  if ((r + 1) * P.NC <= m) ++r;
  return r;
}

// Number of entries of a[0, n) that are <= x, for nondecreasing a.
__device__ __forceinline__ int count_le(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// A decoded item in 16 bytes: kind << 28 | b << 15 | row << 9 | chunk,
// the drafted token of the row (or -1), log2(e)/T (0: greedy), draft length.
__device__ __forceinline__ uint4 pack_item(int kind, int b, int row, int c, int x, float sT, int n) {
  return make_uint4((static_cast<uint32_t>(kind) << 28) | (static_cast<uint32_t>(b) << 15) |
                        (static_cast<uint32_t>(row) << 9) | static_cast<uint32_t>(c),
                    static_cast<uint32_t>(x), __float_as_uint(sT), static_cast<uint32_t>(n));
}
__device__ __forceinline__ Item unpack_item(uint4 e) {
  Item it;
  it.kind = static_cast<int>((e.x >> 28) & 3u);
  it.b = static_cast<int>((e.x >> 15) & 0x3FFu);
  it.row = static_cast<int>((e.x >> 9) & 0x3Fu);
  it.c = static_cast<int>(e.x & 0x1FFu);
  it.x = static_cast<int>(e.y);
  it.sT = __uint_as_float(e.z);
  it.n = static_cast<int>(e.w);
  it.prm = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  return it;
}

// One lane: the item of ticket t < pl.total, packed: tickets run request
// by request, row slot by row slot, chunk by chunk.
__device__ uint4 decode_ticket(const Params& P, const Plan& pl, int t) {
  const bool second = t >= pl.total1;
  const int t2 = second ? t - pl.total1 : t;
  const int r = div_nc(P, t2);
  const int b = count_le(second ? pl.rb2 : pl.rb, P.B, r) - 1;
  const int c = t2 - r * P.NC;
  const int info = pl.info[b];
  const bool sampled = (info & 0x80) != 0;
  // the request's row slot (slots 0 and 1 are the position-0 pair of a
  // request with draft rows, read in the second pass)
  const int slot = second ? r - pl.rb2[b] : r - pl.rb[b] + (two_rows(P, sampled) ? 2 : 0);
  const int n = info & 0x3F;
  const float sT = sampled ? temp_scale(request_T(P, b)) : 0.0f;
  const bool both = two_rows(P, sampled);
  const int row = slot_row(slot, both, n, P.K);
  int x = -1;   // the drafted token whose logit this row's chunks record
  if (both && slot < 2 * n) x = __ldg(P.draft_tokens + static_cast<size_t>(b) * P.K + (slot >> 1));
  else if (sampled && P.mode == kModeOnehot && slot < n)
    x = __ldg(P.draft_tokens + static_cast<size_t>(b) * P.K + slot);
  return pack_item(kItemA, b, row, c, x, sT, n);
}
// ---------------------------------------------------------------- chunk reductions

// Whole warp: argmax of a stats chunk, lowest index on ties.  Each lane
// keeps its maximum and the first of its vectors holding it (its vectors
// taken in increasing order); the warp's first vector holding the maximum
// is then searched once.
template <int DT>
__device__ __forceinline__ float2 chunk_argmax(const unsigned char* slot, const Chunk& k, int lane) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec;
  const Vecs vs = vecs_of<DT>(k);
  const uint4* vec = reinterpret_cast<const uint4*>(slot);
  float best = -INFINITY;
  int bestv = INT_MAX;
  if (lane == 0 && vs.va >= 0) {
    float v[CH];
    masked_vec<DT>(slot, vs, k, vs.va, v);
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < CH; ++q) m = fmaxf(m, v[q]);
    if (m > best) {
      best = m;
      bestv = vs.va;
    }
  }
  int j = vs.vf0 + lane;
  for (; j + 32 < vs.vf1; j += 64) {
    const float m0 = E::vec_max(vec[j]);
    const float m1 = E::vec_max(vec[j + 32]);
    if (m0 > best) {
      best = m0;
      bestv = j;
    }
    if (m1 > best) {
      best = m1;
      bestv = j + 32;
    }
  }
  if (j < vs.vf1) {
    const float m0 = E::vec_max(vec[j]);
    if (m0 > best) {
      best = m0;
      bestv = j;
    }
  }
  if (lane == 1 && vs.vb >= 0) {
    float v[CH];
    masked_vec<DT>(slot, vs, k, vs.vb, v);
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < CH; ++q) m = fmaxf(m, v[q]);
    if (m > best) {
      best = m;
      bestv = vs.vb;
    }
  }
  const float W = warp_max(best);
  if (!(W > -INFINITY)) return make_float2(W, __int_as_float(k.e_lo));   // all -inf (or empty)
  const int vstar = warp_min_int(best == W ? bestv : INT_MAX);
  int idx = INT_MAX;
  if (lane == 0) {
    float v[CH];
    masked_vec<DT>(slot, vs, k, vstar, v);
#pragma unroll
    for (int q = CH - 1; q >= 0; --q)
      if (v[q] == W) idx = vs.e_base + vstar * CH + q;
  }
  idx = __shfl_sync(0xffffffffu, idx, 0);
  return make_float2(W, __int_as_float(idx));
}

// Whole warp: (max, sum of exp((z - max)/T)) of a stats chunk.  The max
// first, then exponents fma(z, sT, -c) against c = fl(max sT); the rounding
// of c is taken out once at the end.
template <int DT>
__device__ __forceinline__ float2 chunk_softmax(const unsigned char* slot, const Chunk& k, float sT, int lane) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec;
  const Vecs vs = vecs_of<DT>(k);
  const uint4* vec = reinterpret_cast<const uint4*>(slot);
  float ev[CH];
  const int my_edge = lane == 0 ? vs.va : (lane == 1 ? vs.vb : -1);
  if (my_edge >= 0) masked_vec<DT>(slot, vs, k, my_edge, ev);
  typename E::MaxAcc acc;
#pragma unroll 4
  for (int j = vs.vf0 + lane; j < vs.vf1; j += 32) acc.add(vec[j]);
  float m = acc.value();
  if (my_edge >= 0) {
#pragma unroll
    for (int q = 0; q < CH; ++q) m = fmaxf(m, ev[q]);
  }
  const float M = warp_max(m);
  if (!(M > -INFINITY)) return make_float2(M, 0.0f);
  const float c = __fmul_rn(M, sT);
  // eight independent sums s_0 .. s_7 (element q of a vector into s_(q mod
  // 8), the second vector of a step after the first), two vectors per step,
  // so the exponentials and the adds of different elements overlap; the
  // sums are kept in pairs (s_2i, s_2i+1) and formed with the two-wide
  // instructions: 2^(z s - c) of two elements per fma, two sums per add
  const f32x2 sT2 = pk2(sT, sT), nc2 = pk2(-c, -c);
  f32x2 s2[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) s2[q] = pk2(0.0f, 0.0f);
  auto add_pair = [&](f32x2& acc, float z0, float z1) {
    float x0, x1;
    up2(fma2(pk2(z0, z1), sT2, nc2), x0, x1);
    acc = add2(acc, pk2(ex2(x0), ex2(x1)));
  };
  int j = vs.vf0 + lane;
#pragma unroll 2
  for (; j + 32 < vs.vf1; j += 64) {
    float a[CH], b[CH];
    E::unpack(vec[j], a);
    E::unpack(vec[j + 32], b);
#pragma unroll
    for (int q = 0; q < CH; q += 2) {
      add_pair(s2[(q & 7) >> 1], a[q], a[q + 1]);
      add_pair(s2[((q + CH) & 7) >> 1], b[q], b[q + 1]);
    }
  }
  if (j < vs.vf1) {
    float a[CH];
    E::unpack(vec[j], a);
#pragma unroll
    for (int q = 0; q < CH; q += 2) add_pair(s2[(q & 7) >> 1], a[q], a[q + 1]);
  }
  if (my_edge >= 0) {
#pragma unroll
    for (int q = 0; q < CH; q += 2) add_pair(s2[(q & 7) >> 1], ev[q], ev[q + 1]);
  }
  float s[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) up2(s2[q], s[2 * q], s[2 * q + 1]);
  const float S = warp_sum(__fadd_rn(__fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3])),
                                     __fadd_rn(__fadd_rn(s[4], s[5]), __fadd_rn(s[6], s[7]))));
  return make_float2(M, __fmul_rn(S, ex2(-__fmaf_rn(M, sT, -c))));
}

// Final-draw weight of one element, scaled by S_p: the residual
// (p - q)+ = max(2^((z - Mp) s) - (S_p/S_q) 2^((y - Mq) s), 0), or p =
// 2^((z - Mp) s) (s = log2(e)/T).  A target logit of -inf (or outside the
// chunk, where slots read -inf) weighs 0; the max with 0 also sends NaN to 0.
__device__ __forceinline__ float weight(float zp, float zq, bool residual, const float4& prm) {
  const float ep = scaled_exp(zp, prm.x, prm.z);
  return fmaxf(residual ? __fmaf_rn(-prm.w, scaled_exp(zq, prm.y, prm.z), ep) : ep, 0.0f);
}

// weight() of two elements at once, residual form, with the two-wide
// instructions: each half is rounded exactly as weight() rounds it.
__device__ __forceinline__ void weight_pair(float zp0, float zp1, float zq0, float zq1,
                                            const float4& prm, float& w0, float& w1) {
  const f32x2 s2 = pk2(prm.z, prm.z);
  float a0, a1, b0, b1;
  up2(mul2(sub2(pk2(zp0, zp1), pk2(prm.x, prm.x)), s2), a0, a1);
  up2(mul2(sub2(pk2(zq0, zq1), pk2(prm.y, prm.y)), s2), b0, b1);
  float r0, r1;
  up2(fma2(pk2(ex2(b0), ex2(b1)), pk2(-prm.w, -prm.w), pk2(ex2(a0), ex2(a1))), r0, r1);
  w0 = fmaxf(r0, 0.0f);
  w1 = fmaxf(r1, 0.0f);
}

// Final-draw weights of vector j of a chunk staged in a slot (target part
// at slot byte 0, draft part at kDraftOff).  The draw items and the final
// search both form weights here, so their sums agree bit for bit.
template <int DT>
__device__ __forceinline__ void vector_weights(const unsigned char* slot, const Vecs& vs,
                                               const Chunk& kp, const Chunk& kq, bool residual,
                                               bool same, const float4& prm, int j, float* w) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec, eb = E::kBytes;
  const int e0 = vs.e_base + j * CH;
  if (!(e0 + CH > kp.e_lo && e0 < kp.e_hi)) {
#pragma unroll
    for (int q = 0; q < CH; ++q) w[q] = 0.0f;
    return;
  }
  const unsigned char* qbuf = slot + kDraftOff;
  float vp[CH], vq[CH];
  if (e0 >= kp.e_lo && e0 + CH <= kp.e_hi) E::unpack(reinterpret_cast<const uint4*>(slot)[j], vp);
  else masked_vec<DT>(slot, vs, kp, j, vp);
  if (residual) {
    if (same) {
      E::unpack(reinterpret_cast<const uint4*>(qbuf)[j], vq);
    } else {
#pragma unroll
      for (int q = 0; q < CH; ++q) {
        const int e = e0 + q;
        vq[q] = (e >= kq.e_lo && e < kq.e_hi) ? E::load(qbuf + kq.off0 + e * eb) : 0.0f;
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < CH; ++q) vq[q] = 0.0f;
  }
  if (residual) {
#pragma unroll
    for (int q = 0; q < CH; q += 2) weight_pair(vp[q], vp[q + 1], vq[q], vq[q + 1], prm, w[q], w[q + 1]);
  } else {
#pragma unroll
    for (int q = 0; q < CH; ++q) w[q] = weight(vp[q], 0.0f, false, prm);
  }
}

// Whole warp: the final draw's token inside a chunk staged in a slot.
// `tau` is the target mass left for this chunk; sweeps (32 vectors each)
// are summed in order (each lane's elements, then across the warp), then
// lanes in order, then the lane's elements.  Rounding that leaves tau beyond the chunk's mass
// falls on the chunk's last positive element.  -1 if nothing weighs > 0.
template <int DT>
__device__ int draw_in_slot(const unsigned char* slot, const Chunk& kp, const Chunk& kq,
                            bool residual, const float4& prm, float tau, int nsw, int lane) {
  constexpr int CH = Elt<DT>::kPerVec;
  const Vecs vs = vecs_of<DT>(kp);
  const bool same = kq.off0 == kp.off0;
  int found = -1, last = -1;
  float tau_s = 0.0f, acc = 0.0f;
  for (int s = 0; s < nsw && found < 0; ++s) {
    float w[CH];
    vector_weights<DT>(slot, vs, kp, kq, residual, same, prm, s * 32 + lane, w);
    float s0 = 0.0f;
#pragma unroll
    for (int q = 0; q < CH; ++q) s0 = __fadd_rn(s0, w[q]);
    const float sw = warp_sum(s0);
    if (sw > 0.0f) {
      if (__fadd_rn(acc, sw) > tau) {
        found = s;
        tau_s = __fsub_rn(tau, acc);
      }
      last = s;
    }
    acc = __fadd_rn(acc, sw);
  }
  if (found < 0) {
    if (last < 0) return -1;
    found = last;
    tau_s = INFINITY;   // the sweep's last positive lane and element
  }
  const int j = found * 32 + lane;
  float w[CH];
  vector_weights<DT>(slot, vs, kp, kq, residual, same, prm, j, w);
  float sum = 0.0f;
#pragma unroll
  for (int q = 0; q < CH; ++q) sum = __fadd_rn(sum, w[q]);
  const float sincl = warp_incl_scan(sum, lane);
  const unsigned hit = __ballot_sync(0xffffffffu, sum > 0.0f && sincl > tau_s);
  const unsigned pos = __ballot_sync(0xffffffffu, sum > 0.0f);
  const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  if (l < 0) return -1;
  const float excl = __shfl_sync(0xffffffffu, __fsub_rn(sincl, sum), l);
  int tok = -1;
  if (lane == l) {
    const float tau3 = __fsub_rn(tau_s, excl);
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
    tok = vs.e_base + j * CH + pick;
  }
  return __shfl_sync(0xffffffffu, tok, l);
}

// ---------------------------------------------------------------- sweep sums

constexpr int kChunkSweeps = kChunkBytes / 512;   // 512-byte sweeps of a stats chunk

// Whole warp: N values per lane (N = 8 or 16) to their sums over the warp,
// halving the values a lane holds at each exchange: lane l ends with the
// sum of value l >> (5 - log2 N) (2 N - 1 shuffles instead of 5 N).
template <int N>
__device__ __forceinline__ float sweep_totals(float (&v)[N], int lane) {
  static_assert(N == 8 || N == 16, "8 or 16 values");
  int o = 16;
#pragma unroll
  for (int h = N / 2; h >= 1; h /= 2) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
    o >>= 1;
  }
#pragma unroll
  for (; o >= 1; o >>= 1) v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
  return v[0];
}

// Whole warp: the residual mass of a piece pair in a slot, sweep by sweep
// (weights formed by vector_weights, as the search forms them).  Returns the piece's total; `mine`
// gets the sum of sweep lane >> 2 (lanes 4 s hold sweep s).
template <int DT>
__device__ float piece_sweeps(const unsigned char* slot, const Chunk& kp, const Chunk& kq,
                              const float4& prm, int lane, float& mine) {
  constexpr int CH = Elt<DT>::kPerVec;
  static_assert(kDrawSweeps <= 8, "sweeps of a piece fit the exchange");
  const Vecs vs = vecs_of<DT>(kp);
  const bool same = kq.off0 == kp.off0;
  float t[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) t[s] = 0.0f;
  float all = 0.0f;
#pragma unroll
  for (int s = 0; s < kDrawSweeps; ++s) {
    float w[CH];
    vector_weights<DT>(slot, vs, kp, kq, true, same, prm, s * 32 + lane, w);
    f32x2 ab = pk2(0.0f, 0.0f);   // even and odd elements' sums
#pragma unroll
    for (int q = 0; q < CH; q += 2) ab = add2(ab, pk2(w[q], w[q + 1]));
    float a, b;
    up2(ab, a, b);
    t[s] = __fadd_rn(a, b);
    all = __fadd_rn(all, t[s]);
  }
  mine = sweep_totals<8>(t, lane);
  return warp_sum(all);
}

// Values of slot vector j of chunk k read from global memory (the slot's
// byte 0 is k.g0), -inf outside [e_lo, e_hi); a whole vector is read at
// once when it lies inside the tensor's aligned range [lo, hi).
template <int DT>
__device__ __forceinline__ void global_vec(const Chunk& k, uintptr_t lo, uintptr_t hi, int j,
                                           float* v) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec, eb = E::kBytes;
  const int e0 = -k.off0 / eb + j * CH;
  const uintptr_t a = k.g0 + static_cast<uintptr_t>(j) * 16;
  if (e0 >= k.e_lo && e0 + CH <= k.e_hi && a >= lo && a + 16 <= hi) {
    E::unpack(__ldg(reinterpret_cast<const uint4*>(a)), v);
    return;
  }
#pragma unroll
  for (int q = 0; q < CH; ++q) {
    const int e = e0 + q;
    v[q] = (e >= k.e_lo && e < k.e_hi) ? E::ldg(reinterpret_cast<const unsigned char*>(a + q * eb))
                                        : -INFINITY;
  }
}

// The same elements of another row (a draft row at `row`): element e at
// row + e * elt.  Elements outside [e_lo, e_hi) read 0.
template <int DT>
__device__ __forceinline__ void global_vec_at(uintptr_t row, uintptr_t lo, uintptr_t hi, int e0,
                                              int e_lo, int e_hi, float* v) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec, eb = E::kBytes;
  const uintptr_t a = row + static_cast<intptr_t>(e0) * eb;
  if (e0 >= e_lo && e0 + CH <= e_hi && (a & 15) == 0 && a >= lo && a + 16 <= hi) {
    E::unpack(__ldg(reinterpret_cast<const uint4*>(a)), v);
    return;
  }
#pragma unroll
  for (int q = 0; q < CH; ++q) {
    const int e = e0 + q;
    v[q] = (e >= e_lo && e < e_hi) ? E::ldg(reinterpret_cast<const unsigned char*>(a + q * eb))
                                   : 0.0f;
  }
}

// Whole warp: the first of n consecutive masses (lane i < n holds mass i)
// whose running total exceeds tau; rounding that leaves tau beyond the
// total falls on the last positive one.  rem gets tau less the masses
// before it.  -1: nothing positive.
__device__ __forceinline__ int pick_lane(float mine, int n, float tau, int lane, float& rem) {
  const float x = lane < n ? mine : 0.0f;
  const float incl = warp_incl_scan(x, lane);
  const unsigned hit = __ballot_sync(0xffffffffu, x > 0.0f && incl > tau);
  const unsigned pos = __ballot_sync(0xffffffffu, x > 0.0f);
  const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  if (l < 0) return -1;
  rem = __fsub_rn(tau, __shfl_sync(0xffffffffu, __fsub_rn(incl, x), l));
  return l;
}

// Whole warp: the element of one sweep whose running weight first exceeds
// tau (lane l holds the weights w[] of vector 32 s + l, first element e0);
// rounding that leaves tau beyond the sweep falls on its last positive
// element.  -1: nothing positive.
template <int CH>
__device__ __forceinline__ int pick_in_sweep(const float* w, float tau, int e0, int lane) {
  float sum = 0.0f;
#pragma unroll
  for (int q = 0; q < CH; ++q) sum = __fadd_rn(sum, w[q]);
  float rem;
  const int l = pick_lane(sum, 32, tau, lane, rem);
  if (l < 0) return -1;
  int tok = -1;
  if (lane == l) {
    float run = 0.0f;
    int pick = -1, lastq = -1;
#pragma unroll
    for (int q = 0; q < CH; ++q) {
      if (w[q] > 0.0f) {
        run = __fadd_rn(run, w[q]);
        if (pick < 0 && run > rem) pick = q;
        lastq = q;
      }
    }
    tok = e0 + (pick < 0 ? lastq : pick);
  }
  return __shfl_sync(0xffffffffu, tok, l);
}


// ---------------------------------------------------------------- draws

// Whole warp: the chunk holding mass u * W of a draw, chunk masses
// mass[c * stride], c in [0, n), in shared memory (lane l sums chunks
// [l m, l m + m) in order,
// then the lanes are scanned).  Returns the chunk and, in rem, the target
// mass left inside it; rounding that leaves the target beyond the total
// falls on the last chunk with positive mass.  Sets W to the total.  -1:
// no mass at all.
__device__ int pick_chunk(const float* mass, int n, float u, int lane, float& W, float& rem,
                          int stride = 1) {
  const int m = (n + 31) / 32;
  const int c0 = min(n, lane * m), c1 = min(n, c0 + m);
  float lane_tot = 0.0f;
  for (int c = c0; c < c1; ++c) lane_tot = __fadd_rn(lane_tot, mass[c * stride]);
  const float incl = warp_incl_scan(lane_tot, lane);
  W = __shfl_sync(0xffffffffu, incl, 31);
  const float excl = __fsub_rn(incl, lane_tot);
  const float tau = __fmul_rn(u, W);
  const unsigned hit = __ballot_sync(0xffffffffu, lane_tot > 0.0f && incl > tau);
  const unsigned pos = __ballot_sync(0xffffffffu, lane_tot > 0.0f);
  const int ol = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  if (ol < 0) return -1;
  int chunk = -1;
  float r = 0.0f;
  if (lane == ol) {
    float acc = excl, last_acc = excl;
    int last_c = -1;
    for (int c = c0; c < c1 && chunk < 0; ++c) {
      const float t = mass[c * stride];
      if (t > 0.0f) {
        if (__fadd_rn(acc, t) > tau) {
          chunk = c;
          r = __fsub_rn(tau, acc);
        }
        last_c = c;
        last_acc = acc;
      }
      acc = __fadd_rn(acc, t);
    }
    if (chunk < 0) {
      chunk = last_c;
      r = __fsub_rn(tau, last_acc);
    }
  }
  rem = __shfl_sync(0xffffffffu, r, ol);
  return __shfl_sync(0xffffffffu, chunk, ol);
}

// Whole warp (control): copies chunk c (of size CB) of target row rp, and
// for a residual the matching draft elements of row rq, into the control
// warp's buffer with bulk copies, and waits (bounded) for them.
// ---------------------------------------------------------------- agents

// A warp's ring: slot s of kSlotBytes at ring + s * kSlotBytes, completing
// on bar[s]; bit s of ph is the parity slot s waits for next.  A slot whose
// item is consumed serves as the warp's scratch until it is refilled.
struct Agent {
  AgentSmem* A;
  unsigned char* ring;
  uint32_t ph;
  int lane;
  __device__ unsigned char* slot(int s) const { return ring + static_cast<size_t>(s) * kSlotBytes; }
};

template <int DT>
__device__ __forceinline__ uintptr_t target_row(const Params& P, int b, int t) {
  return row_addr<DT>(P.target, static_cast<size_t>(b) * (P.K + 1) + t, P.V);
}
template <int DT>
__device__ __forceinline__ uintptr_t draft_row(const Params& P, int b, int t) {
  return row_addr<DT>(P.draft, static_cast<size_t>(b) * P.K + t, P.V);
}
template <int DT>
__device__ __forceinline__ uintptr_t record_row_addr(const Params& P, int b, int row) {
  return row > P.K ? draft_row<DT>(P, b, row - P.K - 1) : target_row<DT>(P, b, row);
}

// Whole warp: waits (bounded) for slot s's copies and flips its parity.
__device__ __forceinline__ bool wait_slot(const Params& P, Agent& ag, int s) {
  const bool ok = warp_wait(&ag.A->bar[s], (ag.ph >> s) & 1u);
  ag.ph ^= 1u << s;
  if (!ok && ag.lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
  return ok;
}

// Lane 0: stages an item into slot s (descriptor, then the bulk copies).
template <int DT>
__device__ void issue(const Params& P, Agent& ag, int s, const Item& it) {
  unsigned char* slot = ag.slot(s);
  uint64_t* bar = &ag.A->bar[s];
  ag.A->item[s] = it;
  uintptr_t src0 = 0, src1 = 0;
  uint32_t n0 = 0, n1 = 0;
  unsigned char *dst0 = slot, *dst1 = slot;
  if (it.kind != kItemR) {
    const bool is_draft = it.row > P.K;
    const Chunk k = chunk_of<DT>(record_row_addr<DT>(P, it.b, it.row), P.V, it.c, kChunkBytes);
    n0 = bulk_span<DT>(k, is_draft ? P.d_lo : P.t_lo, is_draft ? P.d_hi : P.t_hi, &src0);
    if (n0) dst0 = slot + (src0 - k.g0);
  } else {
    const Chunk kp = chunk_of<DT>(target_row<DT>(P, it.b, it.row), P.V, it.c, kDrawBytes);
    n0 = bulk_span<DT>(kp, P.t_lo, P.t_hi, &src0);
    if (n0) dst0 = slot + (src0 - kp.g0);
    const Chunk kq = draft_part<DT>(draft_row<DT>(P, it.b, it.row), kp);
    n1 = bulk_span<DT>(kq, P.d_lo, P.d_hi, &src1);
    if (n1) dst1 = slot + kDraftOff + (src1 - kq.g0);
  }
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(bar, n0 + n1);
  const uint64_t pol = l2_evict_first();
  if (n0) bulk_copy_g2s(dst0, src0, n0, bar, pol);
  if (n1) bulk_copy_g2s(dst1, src1, n1, bar, pol);
}

// Whole warp: copies chunk c (size CB) of target row rp, and for a residual
// the same elements of draft row rq, into scratch slot s and waits for them.
template <int DT>
__device__ bool fetch(const Params& P, Agent& ag, int s, uintptr_t rp, uintptr_t rq, int c, int CB,
                      bool residual, Chunk& kp, Chunk& kq) {
  unsigned char* slot = ag.slot(s);
  kp = chunk_of<DT>(rp, P.V, c, CB);
  kq = residual ? draft_part<DT>(rq, kp) : kp;
  __syncwarp();   // every lane is done with the scratch
  if (ag.lane == 0) {
    uint64_t* bar = &ag.A->bar[s];
    uintptr_t s0 = 0, s1 = 0;
    const uint32_t n0 = bulk_span<DT>(kp, P.t_lo, P.t_hi, &s0);
    const uint32_t n1 = residual ? bulk_span<DT>(kq, P.d_lo, P.d_hi, &s1) : 0u;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, n0 + n1);
    const uint64_t pol = l2_evict_first();
    if (n0) bulk_copy_g2s(slot + (s0 - kp.g0), s0, n0, bar, pol);
    if (n1) bulk_copy_g2s(slot + kDraftOff + (s1 - kq.g0), s1, n1, bar, pol);
  }
  const bool ok = wait_slot(P, ag, s);
  fix_edges<DT>(kp, P.t_lo, P.t_hi, slot, ag.lane);
  if (residual) fix_edges<DT>(kq, P.d_lo, P.d_hi, slot + kDraftOff, ag.lane);
  return ok;
}

// ---------------------------------------------------------------- records

// Whole warp: chunk masses of a draw from p (one row's records rescaled to
// the row maximum Mp) into scratch.
__device__ __forceinline__ void p_masses(const uint2* rec, int NC, float Mp, float sT, float* mass,
                                         int lane) {
  __syncwarp();
  for (int c = lane; c < NC; c += 32) {
    const uint2 r = __ldcg(rec + c);
    const float m = __uint_as_float(r.x);
    mass[c] = m > -INFINITY ? __fmul_rn(__uint_as_float(r.y), scaled_exp(m, Mp, sT)) : 0.0f;
  }
  __syncwarp();
}

// ---------------------------------------------------------------- decisions

constexpr int kMaxRows = 2 * SPECV_MAX_DRAFT + 1 > kMaxTreeNodes ? 2 * SPECV_MAX_DRAFT + 1
                                                                  : kMaxTreeNodes;
constexpr int kDecideRecs = 2048;   // records a decide CTA stages at once (in batches of 1024)
constexpr int kDecideBuf = kDecideRecs > kDecideWarps * kMaxChunks ? kDecideRecs
                                                                    : kDecideWarps * kMaxChunks;

// One lane: a listed draw's record, written / read as two 16-byte words.
__device__ __forceinline__ void store_req(Req* p, int b, int j, float aux, int chunk, float4 prm) {
  *reinterpret_cast<int4*>(p) = make_int4(b, j, __float_as_int(aux), chunk);
  p->prm = prm;
}
__device__ __forceinline__ Req load_req(const Req* p) {
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  Req r;
  r.b = a.x;
  r.j = a.y;
  r.aux = __int_as_float(a.z);
  r.chunk = a.w;
  r.prm = __ldcg(&p->prm);
  return r;
}

// The decision kernel's shared memory: one request's combined rows.
struct DecideSmem {
  float M[kMaxRows], S[kMaxRows];   // row r: maximum (raw logit) and sum, or the argmax value
  int arg[kMaxRows];                // greedy: the argmax
  float mass[kMaxChunks];           // a sampled request's row n: chunk masses of the bonus draw
  int x[SPECV_MAX_DRAFT];           // the request's drafted tokens
  float u[SPECV_MAX_DRAFT + 1];     // its uniforms
  float zp[SPECV_MAX_DRAFT], zq[SPECV_MAX_DRAFT];   // the drafted tokens' logits
  float ur;                         // its resample uniform
  int par[kMaxTreeNodes], tok[kMaxTreeNodes], depth[kMaxTreeNodes];   // tree mode
  alignas(16) uint2 rec[kDecideBuf];   // the request's row records (else each warp's row), staged
};

// One lane: an asynchronous 16-byte copy global -> shared (through L2), and
// the wait for every such copy this lane issued.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Whole warp: n 8-byte records into shared memory, four loads in flight per
// lane before any is stored.
__device__ __forceinline__ void stage_rec(uint2* dst, const uint2* src, int n, int lane) {
  for (int base = 0; base < n; base += 128) {
    uint2 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = base + 32 * k + lane;
      if (i < n) v[k] = __ldcg(src + i);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = base + 32 * k + lane;
      if (i < n) dst[i] = v[k];
    }
  }
  __syncwarp();
}

// Whole warp: combines one row from its NC staged records, a lane per chunk
// (lane c takes chunks c, c + 32, ...): (max, sum of exp((z - max)/T)), or
// at T = 0 (max, lowest index holding it).
__device__ __forceinline__ void combine_row_warp(const uint2* rec, int NC, bool greedy, float sT,
                                                 int lane, float& M, float& S, int& arg) {
  float m = -INFINITY;
  int idx = INT_MAX;
  for (int c = lane; c < NC; c += 32) {
    const uint2 r = rec[c];
    const float v = __uint_as_float(r.x);
    if (v > m) {   // chunks in increasing order: the first chunk holding a lane's maximum
      m = v;
      idx = static_cast<int>(r.y);
    }
  }
  M = warp_max(m);
  S = 0.0f;
  arg = INT_MAX;
  if (greedy) {
    arg = warp_min_int(m == M ? idx : INT_MAX);
    return;
  }
  float s = 0.0f;
  if (M > -INFINITY) {
    for (int c = lane; c < NC; c += 32) {
      const uint2 r = rec[c];
      const float v = __uint_as_float(r.x);
      if (v > -INFINITY) s = __fadd_rn(s, __fmul_rn(__uint_as_float(r.y), scaled_exp(v, M, sT)));
    }
  }
  S = warp_sum(s);
}

// One group of 8 lanes (sub = lane & 7; every lane of the warp calls it):
// combines a row from its NC staged records, chunks c = sub, sub + 8, ...;
// a group with valid false takes no records.
__device__ __forceinline__ void combine_row_group(const uint2* rec, int NC, bool valid, bool greedy,
                                                  float sT, int sub, float& M, float& S,
                                                  int& arg) {
  const int nc = valid ? NC : 0;
  float m = -INFINITY;
  int idx = INT_MAX;
  for (int c = sub; c < nc; c += 8) {
    const uint2 r = rec[c];
    const float v = __uint_as_float(r.x);
    if (v > m) {   // chunks in increasing order: the first chunk holding a lane's maximum
      m = v;
      idx = static_cast<int>(r.y);
    }
  }
  M = m;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  int a = m == M ? idx : INT_MAX;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
  arg = a;
  float s = 0.0f;
  if (!greedy && M > -INFINITY) {
    for (int c = sub; c < nc; c += 8) {
      const uint2 r = rec[c];
      const float v = __uint_as_float(r.x);
      if (v > -INFINITY) s = __fadd_rn(s, __fmul_rn(__uint_as_float(r.y), scaled_exp(v, M, sT)));
    }
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  S = s;
}

// Whole CTA: decides request b from the stats kernel's records and writes
// its outputs.  The CTA's warps combine the request's rows (target rows
// t <= n, draft rows t < n when sampled); warp 0 then takes the decision.
// Greedy: the argmax of target rows t <= n against the drafts.  Sampled:
// the left-to-right test u_t q(x_t) < p(x_t) in log2 form; every draft
// accepted picks the bonus draw's chunk from row n's records and lists the
// request for a bonus walk; a rejection at j stores the residual draw's
// parameters and lists the request for the residual draw.  Either list's
// kernel writes out_tokens[b, n] / out_tokens[b, j].
// A decide CTA's view of request b's own inputs (the caller's buffers):
// length, temperature, their status bits, and for the threads of warp 0 a
// drafted token (lane t < n), a uniform (lane t <= n), the resample uniform
// (lane 0).  Read before waiting on the stats kernel.
struct DecideIn {
  int n, bad, x;
  float T, u, ur;
};

__device__ __forceinline__ DecideIn decide_inputs(const Params& P, int b) {
  const int tid = threadIdx.x, K = P.K;
  DecideIn in;
  in.n = request_len(P, b);
  in.T = request_T(P, b);
  in.bad = request_bad(P, in.n, in.T);
  in.x = -1;
  in.u = 0.0f;
  in.ur = 0.0f;
  if (!in.bad && tid < 32 && P.mode != kModeTree) {
    if (tid < in.n) in.x = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + tid);
    if (tid <= in.n) in.u = __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + tid);
    if (tid == 0 && P.uniforms_resample) in.ur = __ldg(P.uniforms_resample + b);
  }
  return in;
}

template <int DT, int kSite>
__device__ void bonus_draw(const Params& P, uint4* stage, const Req& r, int lane);

// Warp 0, sampler and one-hot rule: the walk of chunk `chunk` of target row
// `row` made at once (the decision's staged records, used by then, as its
// staging) instead of listed for the residual kernel.  Only the walking
// instance of the decision kernel has it.
template <int DT>
__device__ void walk_now(const Params& P, DecideSmem& D, int b, int row, float rem, int chunk,
                         float Mp, int excl, float sT, int lane) {
  Req r;
  r.b = b;
  r.j = row;
  r.aux = rem;
  r.chunk = chunk;
  r.prm = make_float4(Mp, __int_as_float(excl), sT, 0.0f);
  __syncwarp();
  bonus_draw<DT, 1>(P, reinterpret_cast<uint4*>(D.rec), r, lane);
}

// Warp 0, debug calls only: a sampled request's per-row statistics (lane t
// holds row t's): M_p, S_p, ln p(x_t), M_q, S_q, ln q(x_t).
__device__ __noinline__ void write_row_stats(float* rs, int n, bool both, float Mp, float Sp,
                                             float lp, float Mq, float Sq, float lq, int lane) {
  if (lane <= n) {
    rs[lane * 8 + 0] = Mp;
    rs[lane * 8 + 1] = Sp;
  }
  if (lane < n) {
    rs[lane * 8 + 2] = lp * kLn2;
    if (both) {
      rs[lane * 8 + 3] = Mq;
      rs[lane * 8 + 4] = Sq;
      rs[lane * 8 + 5] = lq * kLn2;
    }
  }
}

// Warp 0: a one-hot draft rejected at j.  The replacement comes from
// (p_j - 1{x_j})+, which is p_j with x_j removed: row j's chunk masses of p
// (from its records, staged or in global memory), less x_j's own weight in
// its chunk, pick the chunk; the request joins the bonus list with that
// chunk and x_j excluded from the walk.  If nothing but x_j weighs (p_j(x_j)
// = 1 in fp32, only through rounding), the draw is from p_j itself.
template <int DT, bool kWalk>
__device__ __noinline__ void onehot_rejection(const Params& P, DecideSmem& D, int b, int j, float Mp, float Sp,
                                 float sT, float ur, bool staged, int x_lane, int lane) {
  const int NC = P.NC;
  const uint2* rec = staged ? D.rec + j * NC
                            : P.part + (static_cast<size_t>(b) * P.R + j) * NC;
  const int x = __shfl_sync(0xffffffffu, x_lane, j);
  const float ex = scaled_exp(D.zp[j], Mp, sT);   // x_j's weight, on the scale of the masses
  const uintptr_t ra = target_row<DT>(P, b, j);
  const int cx = static_cast<int>(((ra & 15) + static_cast<uintptr_t>(x) * Elt<DT>::kBytes) /
                                  kChunkBytes);   // the chunk holding x_j
  __syncwarp();
  for (int c = lane; c < NC; c += 32) {
    const uint2 r = staged ? rec[c] : __ldcg(rec + c);
    const float m = __uint_as_float(r.x);
    float w = m > -INFINITY ? __fmul_rn(__uint_as_float(r.y), scaled_exp(m, Mp, sT)) : 0.0f;
    if (c == cx) w = fmaxf(__fsub_rn(w, ex), 0.0f);
    D.mass[c] = w;
  }
  __syncwarp();
  float W, rem;
  int chunk = pick_chunk(D.mass, NC, ur, lane, W, rem);
  int excl = x;
  if (!(W > 0.0f)) {   // only x_j weighs: draw from p_j with the same uniform
    __syncwarp();
    if (lane == (cx & 31)) D.mass[cx] = fmaxf(__fadd_rn(D.mass[cx], ex), ex);
    __syncwarp();
    chunk = pick_chunk(D.mass, NC, ur, lane, W, rem);
    excl = -1;
  }
  float* rs = P.row_stats ? P.row_stats + static_cast<size_t>(b) * (P.K + 1) * 8 : nullptr;
  if (rs && lane == 0) {
    rs[j * 8 + 6] = excl >= 0 ? __fdiv_rn(W, Sp) : 0.0f;
    if (chunk < 0) rs[j * 8 + 7] = -1.0f;
  }
  if (chunk < 0) {
    if (lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_BAD_ROW);
    write_outputs(P, b, -1, -1, x_lane, lane);
    return;
  }
  if (kWalk) {
    write_outputs(P, b, j, -1, x_lane, lane);
    walk_now<DT>(P, D, b, j, rem, chunk, Mp, excl, sT, lane);
    return;
  }
  if (lane == 0)
    store_req(P.req + (P.B - 1 - atomicAdd(P.header + kHBonus, 1)), b, j, rem, chunk,
              make_float4(Mp, __int_as_float(excl), sT, 0.0f));
  write_outputs(P, b, j, -1, x_lane, lane);   // the bonus walk writes the token
}

// Warp 0, tree mode: greedy verification of request b's token tree.  D.arg
// holds the argmax of every node's row (nodes 0..n).  Node i >= 1 is
// accepted iff its parent is and the parent's argmax is its token; the
// deepest accepted node (lowest index among the deepest) ends the path.
// Writes accepted_len = the path's length, out_tokens = the path's tokens
// then the argmax at its last node, path_nodes = 0 then the path's nodes.
// A malformed tree (a parent not below its node, a token outside [0, V))
// gets -1 throughout and a status bit.
__device__ __noinline__ void tree_decide(const Params& P, DecideSmem& D, int b, int n, int lane) {
  const int N = P.K + 1, V = P.V;
  const size_t o = static_cast<size_t>(b) * N;
  int bad = 0;
  for (int i = lane; i <= n; i += 32) {
    const int par = __ldg(P.parents + o + i);
    const int tok = __ldg(P.draft_tokens + o + i);
    D.par[i] = par;
    D.tok[i] = tok;
    if (i == 0 ? par != -1 : (par < 0 || par >= i || tok < 0 || tok >= V)) bad = 1;
    if (D.arg[i] < 0 || D.arg[i] >= V) bad = 1;
  }
  bad = __any_sync(0xffffffffu, bad);
  __syncwarp();
  int len = -1;
  if (!bad && lane == 0) {
    // nodes in index order: a parent is decided before its children
    int best = 0;
    D.depth[0] = 0;
    for (int i = 1; i <= n; ++i) {
      const int par = D.par[i];
      const bool acc = D.depth[par] >= 0 && D.tok[i] == D.arg[par];
      D.depth[i] = acc ? D.depth[par] + 1 : -1;
      if (acc && D.depth[i] > D.depth[best]) best = i;
    }
    len = D.depth[best];
    for (int v = best, k = len; v != 0; v = D.par[v], --k) {
      P.out_tokens[o + k - 1] = D.tok[v];
      P.path_nodes[o + k] = v;
    }
    P.out_tokens[o + len] = D.arg[best];
    P.path_nodes[o] = 0;
    P.accepted_len[b] = len;
    if (P.row_stats)
      for (int i = 0; i <= n; ++i) {
        P.row_stats[(o + i) * 8 + 0] = D.M[i];
        P.row_stats[(o + i) * 8 + 7] = static_cast<float>(D.arg[i]);
      }
  }
  len = __shfl_sync(0xffffffffu, bad ? -1 : len, 0);
  // the padding after the path (everything, for a malformed tree)
  for (int s = lane; s < N; s += 32) {
    if (s > len) P.out_tokens[o + s] = -1;
    if (s > len) P.path_nodes[o + s] = -1;
  }
  if (bad && lane == 0) {
    P.accepted_len[b] = -1;
    atomicOr(P.header + kHStatus, SPECV_DEV_BAD_TREE);
  }
}

template <int DT, bool kWalk>
__device__ void decide_request(const Params& P, DecideSmem& D, int b, const DecideIn& in) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.K, V = P.V, R = P.R, NC = P.NC;
  const int n = in.n;
  const float T = in.T;
  int bad = in.bad;
  if (bad) {
    if (warp == 0) {
      if (lane == 0) atomicOr(P.header + kHStatus, bad);
      write_outputs(P, b, -1, -1, -1, lane);
    }
    return;
  }
  const bool greedy = !(T > 0.0f);
  const float sT = greedy ? 0.0f : temp_scale(T);
  const bool both = two_rows(P, !greedy);
  const int nt = n + 1, nd = both ? n : 0;
  // The request's records and warp 0's inputs (drafted tokens, uniforms,
  // the drafted tokens' logits) in one batch of loads, every load issued
  // before any is stored; records that do not fit are staged a row at a
  // time per warp below.
  const int nrows = nt + nd;
  const bool all_at_once = nrows * NC <= kDecideRecs;
  {
    float zpf = 0.0f, zqf = 0.0f;
    if (!greedy && tid < n) {
      zpf = __ldcg(P.zx + static_cast<size_t>(b) * R + tid);
      if (both) zqf = __ldcg(P.zx + static_cast<size_t>(b) * R + K + 1 + tid);
    }
    constexpr int kPer = 8;
    constexpr int kBatch = kPer * kDecideWarps * 32;
    if (all_at_once) {
      const uint2* base = P.part + static_cast<size_t>(b) * R * NC;
      for (int i0 = 0; i0 < nrows * NC; i0 += kBatch) {
        uint2 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int i = i0 + k * kDecideWarps * 32 + tid;
          if (i < nrows * NC) {
            const int r = i / NC;
            const int row = r < nt ? r : K + 1 + (r - nt);
            v[k] = __ldcg(base + static_cast<size_t>(row) * NC + (i - r * NC));
          }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int i = i0 + k * kDecideWarps * 32 + tid;
          if (i < nrows * NC) D.rec[i] = v[k];
        }
      }
    }
    if (tid < 32 && P.mode != kModeTree) {
      if (tid < SPECV_MAX_DRAFT) {
        D.x[tid] = in.x;
        D.zp[tid] = zpf;
        D.zq[tid] = zqf;
      }
      if (tid <= SPECV_MAX_DRAFT) D.u[tid] = in.u;
      if (tid == 0) D.ur = in.ur;
    }
  }
  __syncthreads();
  if (all_at_once) {
    // a group of 8 lanes per row, 16 rows at a time
    const int sub = lane & 7;
    for (int base = warp * 4; base < nrows; base += kDecideWarps * 4) {
      const int r = base + (lane >> 3);
      float M, S;
      int arg;
      combine_row_group(D.rec + r * NC, NC, r < nrows, greedy, sT, sub, M, S, arg);
      if (r < nrows) {
        if (sub == 0) {
          D.M[r] = M;
          D.S[r] = S;
          D.arg[r] = arg;
        }
        if (!greedy && r == n) {   // the bonus draw's chunk masses, ready before the decision
          const uint2* rec = D.rec + r * NC;
          for (int c = sub; c < NC; c += 8) {
            const float m = __uint_as_float(rec[c].x);
            D.mass[c] = m > -INFINITY ? __fmul_rn(__uint_as_float(rec[c].y), scaled_exp(m, M, sT)) : 0.0f;
          }
        }
      }
    }
  } else {
    for (int r = warp; r < nrows; r += kDecideWarps) {
      const int row = r < nt ? r : K + 1 + (r - nt);
      float M, S;
      int arg;
      uint2* rec = D.rec + warp * kMaxChunks;
      __syncwarp();
      stage_rec(rec, P.part + (static_cast<size_t>(b) * R + row) * NC, NC, lane);
      combine_row_warp(rec, NC, greedy, sT, lane, M, S, arg);
      if (lane == 0) {
        D.M[r] = M;
        D.S[r] = S;
        D.arg[r] = arg;
      }
      if (!greedy && r == n) {
        for (int c = lane; c < NC; c += 32) {
          const float m = __uint_as_float(rec[c].x);
          D.mass[c] = m > -INFINITY ? __fmul_rn(__uint_as_float(rec[c].y), scaled_exp(m, M, sT)) : 0.0f;
        }
      }
    }
  }
  __syncthreads();
  if (warp != 0) return;
  if (P.mode == kModeTree) {
    tree_decide(P, D, b, n, lane);
    return;
  }
  const int x_lane = lane < n ? D.x[lane] : -1;
  const float u_lane = lane <= n ? D.u[lane] : 0.0f;
  const float ur = D.ur;
  const float zp = lane < n ? D.zp[lane] : 0.0f;
  const float zq = lane < n ? D.zq[lane] : 0.0f;

  float Mp_l = -INFINITY, Sp_l = 0.0f, Mq_l = -INFINITY, Sq_l = 0.0f;
  int g = INT_MAX;
  if (lane < nt) {
    Mp_l = D.M[lane];
    Sp_l = D.S[lane];
    g = D.arg[lane];
  }
  if (lane < nd) {
    Mq_l = D.M[nt + lane];
    Sq_l = D.S[nt + lane];
  }
  if (__any_sync(0xffffffffu, lane < n && (x_lane < 0 || x_lane >= V))) bad |= SPECV_DEV_BAD_TOKEN;
  if (__any_sync(0xffffffffu, lane <= n && !(u_lane >= 0.0f && u_lane < 1.0f)) ||
      !(ur >= 0.0f && ur < 1.0f))
    bad |= SPECV_DEV_BAD_UNIFORM;
  float* rs = P.row_stats ? P.row_stats + static_cast<size_t>(b) * (K + 1) * 8 : nullptr;

  if (greedy) {
    if (!bad) {
      if (rs && lane <= n) {
        rs[lane * 8 + 0] = Mp_l;
        rs[lane * 8 + 7] = static_cast<float>(g);
      }
      const unsigned miss = __ballot_sync(0xffffffffu, lane < n && g != x_lane);
      const int j = miss ? __ffs(miss) - 1 : n;
      const int gj = __shfl_sync(0xffffffffu, g, j);
      if (gj >= 0 && gj < V) {
        write_outputs(P, b, j, gj, x_lane, lane);
        return;
      }
      bad = SPECV_DEV_BAD_ROW;
    }
    if (lane == 0) atomicOr(P.header + kHStatus, bad);
    write_outputs(P, b, -1, -1, x_lane, lane);
    return;
  }

  // every row a sampled request needs must have a finite maximum
  if (!bad && __any_sync(0xffffffffu,
                         (lane < n && !(isfinite(Mp_l) && (!both || isfinite(Mq_l)))) ||
                             (lane == n && !isfinite(Mp_l))))
    bad = SPECV_DEV_BAD_ROW;
  if (bad) {
    if (lane == 0) atomicOr(P.header + kHStatus, bad);
    write_outputs(P, b, -1, -1, x_lane, lane);
    return;
  }
  float lp = 0.0f, lq = 0.0f;
  bool accept = false;
  if (lane < n) {
    lp = __fsub_rn(__fmul_rn(__fsub_rn(zp, Mp_l), sT), __log2f(Sp_l));
    // a one-hot draft's q(x) = 1: accept iff u < p(x)
    lq = both ? __fsub_rn(__fmul_rn(__fsub_rn(zq, Mq_l), sT), __log2f(Sq_l)) : 0.0f;
    accept = __fadd_rn(__log2f(u_lane), lq) < lp;
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < n && !accept);
  const int j = rej ? __ffs(rej) - 1 : n;
  if (rs) write_row_stats(rs, n, both, Mp_l, Sp_l, lp, Mq_l, Sq_l, lq, lane);
  const float Mp = __shfl_sync(0xffffffffu, Mp_l, j);
  const float Sp = __shfl_sync(0xffffffffu, Sp_l, j);
  if (j < n && !both) {
    onehot_rejection<DT, kWalk>(P, D, b, j, Mp, Sp, sT, ur, all_at_once, x_lane, lane);
    return;
  }
  if (j < n) {
    const float Mq = __shfl_sync(0xffffffffu, Mq_l, j);
    const float Sq = __shfl_sync(0xffffffffu, Sq_l, j);
    if (lane == 0) {
      store_req(P.req + atomicAdd(P.header + kHResid, 1), b, j, Sp, __float_as_int(ur),
                make_float4(Mp, Mq, sT, __fdiv_rn(Sp, Sq)));
    }
    write_outputs(P, b, j, -1, x_lane, lane);   // the residual kernel writes the token
    return;
  }
  // every draft accepted: the bonus token from p_n with uniforms[b, n].  The
  // chunk is picked here from row n's chunk masses; the residual kernel
  // walks that chunk to the token and writes out_tokens[b, n].
  const float u = __shfl_sync(0xffffffffu, u_lane, n);
  float W, rem;
  const int chunk = pick_chunk(D.mass, NC, u, lane, W, rem);
  if (rs && lane == 0) {
    rs[n * 8 + 6] = __fdiv_rn(W, Sp);
    if (chunk < 0) rs[n * 8 + 7] = -1.0f;
  }
  if (chunk < 0) {
    if (lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_BAD_ROW);
    write_outputs(P, b, -1, -1, x_lane, lane);
    return;
  }
  if (kWalk) {
    write_outputs(P, b, n, -1, x_lane, lane);
    walk_now<DT>(P, D, b, n, rem, chunk, Mp, -1, sT, lane);
    return;
  }
  if (lane == 0) {
    store_req(P.req + (P.B - 1 - atomicAdd(P.header + kHBonus, 1)), b, n, rem, chunk,
              make_float4(Mp, __int_as_float(-1), sT, 0.0f));   // the bonus list grows down
  }
  write_outputs(P, b, n, -1, x_lane, lane);
}

// Whole warp: vectors jv of chunk kp that the cp.async staging skipped
// (bit jv / 32 of `whole` clear: partly outside the chunk or the tensor's
// aligned range) read element by element into the stage, -inf outside the
// chunk.  Rare (a row's edges), so kept out of line; one instance per
// calling kernel (kSite, as bonus_draw's), so that a second caller leaves
// the residual kernel's register allocation as it was.
template <int DT, int kSite>
__device__ __noinline__ void stage_edges(const Params& P, uint4* stage, const Chunk& kp,
                                         unsigned whole, int lane) {
  constexpr int CH = Elt<DT>::kPerVec;
  for (int s = 0; s < kChunkSweeps; ++s) {
    if ((whole >> s) & 1u) continue;
    float v[CH];
    global_vec<DT>(kp, P.t_lo, P.t_hi, s * 32 + lane, v);
    unsigned char* dst = reinterpret_cast<unsigned char*>(stage + s * 32 + lane);
#pragma unroll
    for (int q = 0; q < CH; ++q) {
      if (DT == SPECV_BF16)
        reinterpret_cast<unsigned short*>(dst)[q] = static_cast<unsigned short>(__float_as_uint(v[q]) >> 16);
      else
        reinterpret_cast<float*>(dst)[q] = v[q];
    }
  }
}

// Whole warp: the bonus token of listed draw r (every draft accepted):
// the decision's chunk of target row n copied into `stage` (16-byte
// aligned, kChunkBytes; the token the draw leaves out, if any, set to
// -inf there), its sweeps' masses of p summed in order, four sweeps at a
// time, until the running total passes the target left at the chunk, then
// the token inside that sweep.  Rounding that leaves the target past the
// chunk's sweeps falls on the last positive one.  Writes out_tokens[b, n], or -1
// throughout (status bit) when nothing is drawn.
// kSite: which kernel calls it (0 the residual kernel, 1 the decision
// kernel's own walks), so that each kernel has its own instance and the
// second caller leaves the residual kernel's compilation as it was.
template <int DT, int kSite = 0>
__device__ void bonus_draw(const Params& P, uint4* stage, const Req& r, int lane) {
  using E = Elt<DT>;
  constexpr int CH = E::kPerVec;
  const int K = P.K, V = P.V;
  const int b = r.b, n = r.j, chunk = r.chunk;
  const float rem = r.aux;
  const float4 prm = r.prm;
  const int excl = __float_as_int(prm.y);   // a token the draw leaves out (-1: none)
  const Chunk kp = chunk_of<DT>(target_row<DT>(P, b, n), V, chunk, kChunkBytes);
  const int e_base = -kp.off0 / E::kBytes;   // the element at stage byte 0
  // every 16-byte vector of the chunk copied at once into the staging area
  // with cp.async; the few partly outside the chunk (row edges) element by
  // element
  unsigned whole = 0u;
#pragma unroll
  for (int s = 0; s < kChunkSweeps; ++s) {
    const int jv = s * 32 + lane;
    const int e0 = e_base + jv * CH;
    const uintptr_t a = kp.g0 + static_cast<uintptr_t>(jv) * 16;
    const bool in = e0 >= kp.e_lo && e0 + CH <= kp.e_hi && a >= P.t_lo && a + 16 <= P.t_hi;
    if (in) cp_async16(stage + jv, reinterpret_cast<const void*>(a));
    whole |= static_cast<unsigned>(in) << s;
  }
  if (__any_sync(0xffffffffu, whole != (1u << kChunkSweeps) - 1u)) stage_edges<DT, kSite>(P, stage, kp, whole, lane);
  cp_async_wait_all();
  __syncwarp();
  if (lane == 0 && excl >= kp.e_lo && excl < kp.e_hi) {
    unsigned char* x = reinterpret_cast<unsigned char*>(stage) + (excl - e_base) * E::kBytes;
    if (DT == SPECV_BF16) *reinterpret_cast<unsigned short*>(x) = 0xFF80u;
    else *reinterpret_cast<float*>(x) = -INFINITY;
  }
  __syncwarp();
  // sweeps in order, four at a time (their sums formed together), until
  // the running mass passes the target; then the token inside the sweep
  static_assert(kChunkSweeps % 4 == 0, "a chunk is whole groups of four sweeps");
  float acc = 0.0f, rem2 = 0.0f;
  int found = -1, last = -1;
#pragma unroll 1
  for (int g = 0; g < kChunkSweeps && found < 0; g += 4) {
    float t4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[CH];
      E::unpack(stage[(g + k) * 32 + lane], v);
      float a = 0.0f;
#pragma unroll
      for (int q = 0; q < CH; ++q) a = __fadd_rn(a, weight(v[q], 0.0f, false, prm));
      t4[k] = a;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) t4[k] = warp_sum(t4[k]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (found >= 0) continue;
      if (t4[k] > 0.0f) {
        if (__fadd_rn(acc, t4[k]) > rem) {
          found = g + k;
          rem2 = __fsub_rn(rem, acc);
          continue;
        }
        last = g + k;
      }
      acc = __fadd_rn(acc, t4[k]);
    }
  }
  if (found < 0 && last >= 0) {   // the last positive sweep, its last positive element
    found = last;
    rem2 = INFINITY;
  }
  int tok = -1;
  if (found >= 0) {
    float v[CH], w[CH];
    E::unpack(stage[found * 32 + lane], v);
#pragma unroll
    for (int q = 0; q < CH; ++q) w[q] = weight(v[q], 0.0f, false, prm);
    tok = pick_in_sweep<CH>(w, rem2, e_base + (found * 32 + lane) * CH, lane);
  }
  if (P.row_stats && lane == 0)
    P.row_stats[(static_cast<size_t>(b) * (K + 1) + n) * 8 + 7] = static_cast<float>(tok);
  if (tok < 0 || tok >= V) {
    if (lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_BAD_ROW);
    write_outputs(P, b, -1, -1, -1, lane);
  } else if (lane == 0) {
    P.out_tokens[static_cast<size_t>(b) * (K + 1) + n] = tok;
  }
  __syncwarp();
}

// Whole warp: starts copying entry e's piece records into slot 0 of the
// warp's ring (cp.async; residual_search waits), when they fit the slot.
__device__ __forceinline__ void stage_pieces(const Params& P, Agent& ag, int e) {
  if (P.NCd * kPieceRec * 4 > kSlotBytes) return;
  const uint4* src = reinterpret_cast<const uint4*>(P.dpc + static_cast<size_t>(e) * P.NCd * kPieceRec);
  uint4* dst = reinterpret_cast<uint4*>(ag.slot(0));
  __syncwarp();   // every lane is done with the scratch
  for (int i = ag.lane; i < P.NCd * kPieceRec / 4; i += 32) cp_async16(dst + i, src + i);
}

// Whole warp: the residual draw of list entry e (record r: request b,
// rejected at row j, the resample uniform): the piece from the piece sums,
// the sweep from that piece's sweep sums, the token from the sweep of both
// rows read again.  A residual of exactly zero mass falls back to drawing
// from p_j with the same uniform (its chunk masses from row j's records,
// the token from one re-read chunk).  Slot 0 of the warp's ring is its
// scratch; stage_pieces(e) has been called.
template <int DT>
__device__ void residual_search(const Params& P, Agent& ag, int e, const Req& r) {
  constexpr int CH = Elt<DT>::kPerVec;
  const int lane = ag.lane, K = P.K, V = P.V, NC = P.NC, NCd = P.NCd;
  const int b = r.b, j = r.j;
  const float4 prm = r.prm;
  const float ur = __int_as_float(r.chunk);
  float* mass = reinterpret_cast<float*>(ag.slot(0));
  const float* pc = P.dpc + static_cast<size_t>(e) * NCd * kPieceRec;
  const bool staged = NCd * kPieceRec * 4 <= kSlotBytes;
  cp_async_wait_all();
  __syncwarp();
  if (!staged) {   // the piece totals alone, gathered
    for (int c = lane; c < NCd; c += 32) mass[c] = __ldcg(pc + c * kPieceRec + kDrawSweeps);
    __syncwarp();
  }
  float W = 0.0f, rem = 0.0f;
  int chunk = staged ? pick_chunk(mass + kDrawSweeps, NCd, ur, lane, W, rem, kPieceRec)
                     : pick_chunk(mass, NCd, ur, lane, W, rem);
  const uintptr_t rp = target_row<DT>(P, b, j);
  int tok = -1;
  if (W > 0.0f) {
    if (chunk >= 0) {
      const float sw = lane < kDrawSweeps ? (staged ? mass[chunk * kPieceRec + lane]
                                                    : __ldcg(pc + chunk * kPieceRec + lane))
                                          : 0.0f;
      float rem2 = 0.0f;
      const int sweep = pick_lane(sw, kDrawSweeps, rem, lane, rem2);
      if (sweep >= 0) {
        const Chunk kp = chunk_of<DT>(rp, V, chunk, kDrawBytes);
        const int jv = sweep * 32 + lane;
        const int e0 = -kp.off0 / Elt<DT>::kBytes + jv * CH;
        float vp[CH], vq[CH], w[CH];
        global_vec<DT>(kp, P.t_lo, P.t_hi, jv, vp);
        global_vec_at<DT>(draft_row<DT>(P, b, j), P.d_lo, P.d_hi, e0, kp.e_lo, kp.e_hi, vq);
#pragma unroll
        for (int q = 0; q < CH; ++q) w[q] = weight(vp[q], vq[q], true, prm);
        tok = pick_in_sweep<CH>(w, rem2, e0, lane);
      }
    }
  } else {
    p_masses(P.part + (static_cast<size_t>(b) * P.R + j) * NC, NC, prm.x, prm.z, mass, lane);
    float Wp;
    chunk = pick_chunk(mass, NC, ur, lane, Wp, rem);
    Chunk kp, kq;
    if (chunk >= 0 && fetch<DT>(P, ag, 0, rp, 0, chunk, kChunkBytes, false, kp, kq))
      tok = draw_in_slot<DT>(ag.slot(0), kp, kq, false, make_float4(prm.x, 0.0f, prm.z, 0.0f),
                             rem, kChunkBytes / 512, lane);
  }
  if (P.row_stats && lane == 0) {
    float* rs = P.row_stats + (static_cast<size_t>(b) * (K + 1) + j) * 8;
    rs[6] = __fdiv_rn(W, r.aux);
    rs[7] = static_cast<float>(tok);
  }
  if (tok < 0 || tok >= V) {
    if (lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_BAD_ROW);
    write_outputs(P, b, -1, -1, -1, lane);
  } else if (lane == 0) {
    P.out_tokens[static_cast<size_t>(b) * (K + 1) + j] = tok;
  }
  __syncwarp();
}

// ---------------------------------------------------------------- programmatic launch

// The next kernel on the stream may start launching (its prologue overlaps
// this kernel's tail; it waits for this kernel's results before reading).
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the previous kernel on the stream has completed and its
// writes are visible.
__device__ __forceinline__ void wait_previous() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- stats kernel

// Whole warp: reduces the chunk in slot s to its record; the chunk holding
// the row's drafted token also records that token's logit.
template <int DT>
__device__ void consume_stats(const Params& P, Agent& ag, int s, const Item& it) {
  const int lane = ag.lane;
  unsigned char* slot = ag.slot(s);
  const bool is_draft = it.row > P.K;
  const Chunk k = chunk_of<DT>(record_row_addr<DT>(P, it.b, it.row), P.V, it.c, kChunkBytes);
  fix_edges<DT>(k, is_draft ? P.d_lo : P.t_lo, is_draft ? P.d_hi : P.t_hi, slot, lane);
  float2 r;
  if (it.sT > 0.0f)
    r = chunk_softmax<DT>(slot, k, it.sT, lane);
  else
    r = chunk_argmax<DT>(slot, k, lane);
  if (lane == 0) {
    const uint64_t keep = l2_evict_last();
    st_keep(P.part + (static_cast<size_t>(it.b) * P.R + it.row) * P.NC + it.c,
            make_uint2(__float_as_uint(r.x), __float_as_uint(r.y)), keep);
    if (it.x >= k.e_lo && it.x < k.e_hi)
      st_keep(P.zx + static_cast<size_t>(it.b) * P.R + it.row,
              Elt<DT>::load(slot + k.off0 + it.x * Elt<DT>::kBytes), keep);
  }
}

// A warp's tickets, decoded 32 at a time (one per lane): the warp's i-th
// ticket is first + i * stride.
struct TicketRun {
  int first, stride, total;
  int base;     // index of the ticket lane 0 holds
  uint4 mine;   // this lane's decoded ticket (base + lane)
};

// Whole warp: the i-th ticket's item (i increasing); false past the last.
__device__ __forceinline__ bool run_item(const Params& P, const Plan& pl, TicketRun& tr, int i,
                                         int lane, Item& it) {
  if (tr.first + i * tr.stride >= tr.total) return false;
  if (i >= tr.base + 32) {
    tr.base = i;
    const int t = tr.first + (i + lane) * tr.stride;
    if (t < tr.total) tr.mine = decode_ticket(P, pl, t);
  }
  const int l = i - tr.base;
  uint4 e;
  e.x = __shfl_sync(0xffffffffu, tr.mine.x, l);
  e.y = __shfl_sync(0xffffffffu, tr.mine.y, l);
  e.z = __shfl_sync(0xffffffffu, tr.mine.z, l);
  e.w = __shfl_sync(0xffffffffu, tr.mine.w, l);
  it = unpack_item(e);
  return true;
}

// Whole warp: one agent of the stats kernel.  Warp g of the grid's G
// streams tickets g, g + G, g + 2 G, ... through its ring, refilling a slot
// as soon as its chunk is reduced.
template <int DT>
__device__ void stats_agent(const Params& P, const Plan& pl, Agent& ag, int g, int G) {
  const int lane = ag.lane;
  TicketRun tr;
  tr.first = g;
  tr.stride = G;
  tr.total = pl.total;
  tr.base = -64;
  tr.mine = make_uint4(0u, 0u, 0u, 0u);
  int issued = 0, consumed = 0;
  for (;;) {
    while (issued - consumed < kSlots) {
      Item it;
      if (!run_item(P, pl, tr, issued, lane, it)) break;
      __syncwarp();
      if (lane == 0) issue<DT>(P, ag, issued % kSlots, it);
      ++issued;
    }
    if (issued == consumed) break;   // no tickets left and nothing in flight
    const int s = consumed % kSlots;
    if (!wait_slot(P, ag, s)) return;
    consume_stats<DT>(P, ag, s, ag.A->item[s]);
    ++consumed;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) stats_kernel(const Params P) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  __shared__ Smem S;
  extern __shared__ __align__(128) unsigned char dyn[];

  if (tid < kAgents * kSlots) {
    mbar_init(&S.ag[tid / kSlots].bar[tid % kSlots], 1);
    mbar_init_fence();
  }
  build_plan(P, S.plan, S.red);   // ends with a CTA barrier; reads the inputs only
  // The previous kernel on the stream (the last one of an earlier call, when
  // calls follow each other) may still run: write nothing before it ends.
  wait_previous();
  allow_dependents();
  if (blockIdx.x == 0 && tid == 0) {   // the lists the decisions fill start empty
    P.header[kHResid] = 0;
    P.header[kHBonus] = 0;
  }

  Agent ag;
  ag.A = &S.ag[warp];
  ag.ring = dyn + static_cast<size_t>(warp) * kSlots * kSlotBytes;
  ag.ph = 0;
  ag.lane = tid & 31;
  stats_agent<DT>(P, S.plan, ag, static_cast<int>(blockIdx.x) * kAgents + warp,
                  static_cast<int>(gridDim.x) * kAgents);

}

// ---------------------------------------------------------------- decide kernel

// kWalk: the sampler and the one-hot rule, whose draws are walks the
// decision makes itself; otherwise walks and residual draws are listed.
template <int DT, bool kWalk>
__global__ void __launch_bounds__(kDecideWarps * 32, 4) decide_kernel(const Params P) {
  __shared__ DecideSmem D;
  // the first request's own inputs are fetched while the stats kernel runs
  int b = static_cast<int>(blockIdx.x);
  DecideIn in = decide_inputs(P, min(b, P.B - 1));
  wait_previous();
  allow_dependents();
  for (; b < P.B; b += gridDim.x) {
    if (b != static_cast<int>(blockIdx.x)) in = decide_inputs(P, b);
    decide_request<DT, kWalk>(P, D, b, in);
    __syncthreads();
  }
}

// ---------------------------------------------------------------- residual kernel

// Whole warp: sums the residual (p - q)+ of the piece pair in slot s,
// sweep by sweep, and stores the piece's sum and its sweep sums.
template <int DT>
__device__ void consume_residual(const Params& P, Agent& ag, int s, const Item& it) {
  const int lane = ag.lane;
  unsigned char* slot = ag.slot(s);
  const Chunk kp = chunk_of<DT>(target_row<DT>(P, it.b, it.row), P.V, it.c, kDrawBytes);
  fix_edges<DT>(kp, P.t_lo, P.t_hi, slot, lane);
  const Chunk kq = draft_part<DT>(draft_row<DT>(P, it.b, it.row), kp);
  fix_edges<DT>(kq, P.d_lo, P.d_hi, slot + kDraftOff, lane);
  float mine;
  const float t = piece_sweeps<DT>(slot, kp, kq, it.prm, lane, mine);
  const int e = it.n;   // the request's entry in the list
  float* pr = P.dpc + (static_cast<size_t>(e) * P.NCd + it.c) * kPieceRec;
  if ((lane & 3) == 0 && (lane >> 2) < kDrawSweeps) pr[lane >> 2] = mine;
  if (lane == 0) pr[kDrawSweeps] = t;
}

// One lane: residual item i (entry i / NCd, piece i mod NCd).  An entry
// past the list's B slots is read as the last slot (a decode made before
// the list's length is known; such an item is never used).
__device__ __forceinline__ Item residual_item(const Params& P, int i) {
  Item it;
  const int e = min(i / P.NCd, P.B - 1);
  it.kind = kItemR;
  it.c = i - e * P.NCd;
  it.n = e;
  const Req r = load_req(P.req + e);
  it.b = r.b;
  it.row = r.j;
  it.prm = r.prm;
  it.sT = 0.0f;
  it.x = -1;
  return it;
}

// Whole warp: the warp's k-th residual item (lane k mod 32 decoded it).
__device__ __forceinline__ Item residual_pick(const Item& mine, int l) {
  Item it;
  it.kind = kItemR;
  it.c = __shfl_sync(0xffffffffu, mine.c, l);
  it.n = __shfl_sync(0xffffffffu, mine.n, l);
  it.b = __shfl_sync(0xffffffffu, mine.b, l);
  it.row = __shfl_sync(0xffffffffu, mine.row, l);
  it.prm.x = __shfl_sync(0xffffffffu, mine.prm.x, l);
  it.prm.y = __shfl_sync(0xffffffffu, mine.prm.y, l);
  it.prm.z = __shfl_sync(0xffffffffu, mine.prm.z, l);
  it.prm.w = __shfl_sync(0xffffffffu, mine.prm.w, l);
  it.sT = 0.0f;
  it.x = -1;
  return it;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) residual_kernel(const Params P) {
  __shared__ AgentSmem A[kAgents];
  extern __shared__ __align__(128) unsigned char dyn[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < kAgents * kSlots) {
    mbar_init(&A[tid / kSlots].bar[tid % kSlots], 1);
    mbar_init_fence();
  }
  __syncthreads();
  wait_previous();
  Agent ag;
  ag.A = &A[warp];
  ag.ring = dyn + static_cast<size_t>(warp) * kSlots * kSlotBytes;
  ag.ph = 0;
  ag.lane = lane;
  allow_dependents();
  // The grid's warps in CTA-interleaved order (consecutive positions on
  // different SMs): the bonus draws take positions 0, 1, ..., the residual
  // pieces positions G - 1, G - 2, ..., so both spread over every SM.  A
  // warp's first piece is decoded (its list entry loaded, by lane 0)
  // together with the lists' lengths; an entry past the residual list's end
  // is stale and never used.
  const int G = static_cast<int>(gridDim.x) * kAgents;
  const int pos = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  const int first = G - 1 - pos;   // the warp's pieces: first, first + G, ...
  Item mine{};
  if (lane == 0) mine = residual_item(P, first);
  int base = 0, decoded = 1;       // lanes holding decoded items
  const int count = __ldcg(P.header + kHResid);
  const int nb = __ldcg(P.header + kHBonus);
  const int total = count * P.NCd;
  for (int k = pos; k < nb; k += G)   // a warp each, slot 0 of its ring as staging
    bonus_draw<DT>(P, reinterpret_cast<uint4*>(ag.slot(0)), load_req(P.req + (P.B - 1 - k)), lane);
  if (pos < nb) fence_proxy_async_smem();   // staging writes before bulk copies into the slot
  const int mine_n = first < total ? (total - first + G - 1) / G : 0;
  int issued = 0, consumed = 0;
  for (;;) {
    while (issued - consumed < kSlots && issued < mine_n) {
      if (issued >= base + decoded) {   // decode the next 32 of this warp's items, one per lane
        base = issued;
        decoded = 32;
        const int i = first + (base + lane) * G;
        if (i < total) mine = residual_item(P, i);
      }
      const Item it = residual_pick(mine, issued - base);
      __syncwarp();
      if (lane == 0) issue<DT>(P, ag, issued % kSlots, it);
      ++issued;
    }
    if (issued == consumed) break;
    const int s = consumed % kSlots;
    if (!wait_slot(P, ag, s)) break;
    consume_residual<DT>(P, ag, s, A[warp].item[s]);
    ++consumed;
  }
}

// ---------------------------------------------------------------- search kernel

template <int DT>
__global__ void __launch_bounds__(kDecideWarps * 32) search_kernel(const Params P) {
  __shared__ AgentSmem A[kDecideWarps];
  extern __shared__ __align__(128) unsigned char dyn[];
  const int tid = threadIdx.x, warp = tid >> 5;
  if ((tid & 31) == 0) {
    mbar_init(&A[warp].bar[0], 1);
    mbar_init_fence();
  }
  __syncwarp();
  wait_previous();
  allow_dependents();
  Agent ag;
  ag.A = &A[warp];
  ag.ring = dyn + static_cast<size_t>(warp) * kSlotBytes;
  ag.ph = 0;
  ag.lane = tid & 31;
  // the first entry's records are requested before the list's length is
  // known (entries past it read stale workspace, and are not used)
  const int e0 = static_cast<int>(blockIdx.x) * kDecideWarps + warp;
  Req r = load_req(P.req + min(e0, P.B - 1));
  stage_pieces(P, ag, min(e0, P.B - 1));
  const int count = __ldcg(P.header + kHResid);
  for (int e = e0; e < count; e += gridDim.x * kDecideWarps) {
    if (e != e0) {
      r = load_req(P.req + e);
      stage_pieces(P, ag, e);
    }
    residual_search<DT>(P, ag, e, r);
  }
  cp_async_wait_all();
}

// ---------------------------------------------------------------- post-accept insert

constexpr int kInsertThreads = 1024;

// One CTA: request b = tile base + thread.  Each emits j + 1 tokens when
// j = accepted_len[b] is in [0, K] and its history has room (else nothing,
// with status 1 or 2); cu_emitted is the exclusive prefix of the emitted
// counts over requests (a block-wide scan per tile of 1024, carried from
// tile to tile), and the emitted tokens are written both behind the
// request's history and packed at cu_emitted[b].
__global__ void __launch_bounds__(kInsertThreads) insert_kernel(
    const int32_t* __restrict__ accepted_len, const int32_t* __restrict__ out_tokens, int B, int K1,
    int32_t* seq_lens, int32_t* history, int L, int32_t* next_tokens, int32_t* cu_emitted,
    int32_t* packed, int32_t* status) {
  __shared__ int wsum[kInsertThreads / 32];
  __shared__ int tile_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  for (int base = 0; base < B; base += kInsertThreads) {
    const int b = base + tid;
    int j = -1, s0 = 0, em = 0, st = 0;
    if (b < B) {
      j = accepted_len[b];
      s0 = seq_lens[b];
      if (j < 0 || j >= K1) st = 1;
      else if (s0 < 0 || s0 > L - (j + 1)) st = 2;
      else em = j + 1;
    }
    const int incl = warp_incl_scan_int(em, lane);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = wsum[lane];
      const int wi = warp_incl_scan_int(v, lane);
      wsum[lane] = wi - v;
      if (lane == 31) tile_total = wi;
    }
    __syncthreads();
    const int excl = carry + wsum[warp] + incl - em;
    if (b < B) {
      const int32_t* out = out_tokens + static_cast<size_t>(b) * K1;
      cu_emitted[b] = excl;
      status[b] = st;
      if (em) {
        int32_t* h = history + static_cast<size_t>(b) * L + s0;
        for (int i = 0; i < em; ++i) {
          const int32_t t = out[i];
          h[i] = t;
          packed[excl + i] = t;
        }
        seq_lens[b] = s0 + em;
        next_tokens[b] = out[j];
      } else {
        next_tokens[b] = -1;
      }
      if (b == B - 1) cu_emitted[B] = excl + em;
    }
    carry += tile_total;
    __syncthreads();   // wsum and tile_total are rewritten by the next tile
  }
}

// ---------------------------------------------------------------- host gather

constexpr int kGatherThreads = 512;

// Copies the logit rows the kernels read from page-locked host memory
// (device-visible at ht / hd) into the staging copies dt / dd, with 16-byte
// loads over the host link: target rows t <= n_b and, for a sampled request
// with draft logits, draft rows t < n_b.  Rows are row16 16-byte words (the
// host entry point takes this path only when V * elt is a multiple of 16 and
// every base is 16-byte aligned).  A request that the decision flags (a draft
// length outside 1..K, a bad temperature) gets no rows.  CTA c takes row
// slots c, c + grid, ... of the B * (2K + 1) slots, eight words per thread in
// flight.
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(
    const uint4* __restrict__ ht, const uint4* __restrict__ hd, uint4* __restrict__ dt,
    uint4* __restrict__ dd, const int32_t* __restrict__ draft_len,
    const float* __restrict__ temperature, int B, int K, size_t row16) {
  const int S = 2 * K + 1;
  for (int r = static_cast<int>(blockIdx.x); r < B * S; r += static_cast<int>(gridDim.x)) {
    const int b = r / S, slot = r - b * S;
    const int n = draft_len ? draft_len[b] : K;
    const float T = temperature[b];
    if (n < 1 || n > K || !(T >= 0.0f) || isinf(T)) continue;
    const uint4* src;
    uint4* dst;
    if (slot <= K) {
      if (slot > n) continue;
      const size_t off = (static_cast<size_t>(b) * (K + 1) + slot) * row16;
      src = ht + off;
      dst = dt + off;
    } else {
      const int t = slot - K - 1;
      if (!(T > 0.0f) || hd == nullptr || t >= n) continue;
      const size_t off = (static_cast<size_t>(b) * K + t) * row16;
      src = hd + off;
      dst = dd + off;
    }
    constexpr int kUnroll = 8;
    size_t i = threadIdx.x;
    for (; i + (kUnroll - 1) * kGatherThreads < row16; i += kUnroll * kGatherThreads) {
      uint4 v[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) v[k] = __ldcs(src + i + k * kGatherThreads);
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) dst[i + k * kGatherThreads] = v[k];
    }
    for (; i < row16; i += kGatherThreads) dst[i] = __ldcs(src + i);
  }
}

// ---------------------------------------------------------------- host side


int elt_bytes(specv_dtype dt) { return dt == SPECV_BF16 ? 2 : 4; }

struct Layout {
  size_t header, req, part, zx, dpc, total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Chunks per row for chunk size CB, for any 16-byte phase of the row.
int chunks_per_row(int V, specv_dtype dt, int CB) {
  return static_cast<int>((15 + static_cast<long long>(V) * elt_bytes(dt) + CB - 1) / CB);
}

// Requests per launch sequence: larger batches run as consecutive
// sequences that share the workspace.
int launch_batch(int B) { return B < kPlanMax ? B : kPlanMax; }

Layout ws_layout(int B, int K, int V, specv_dtype dt) {
  const size_t Bl = static_cast<size_t>(launch_batch(B));
  const size_t R = 2 * static_cast<size_t>(K) + 1;
  const size_t NC = chunks_per_row(V, dt, kChunkBytes);
  const size_t NCd = chunks_per_row(V, dt, kDrawBytes);
  Layout L;
  L.header = 0;
  L.req = kHeaderBytes;
  L.part = align256(L.req + sizeof(Req) * Bl);
  L.zx = align256(L.part + sizeof(uint2) * Bl * R * NC);
  L.dpc = align256(L.zx + sizeof(float) * Bl * R);
  L.total = align256(L.dpc + sizeof(float) * Bl * NCd * kPieceRec);
  return L;
}

// Resident CTAs of the stats kernel on the current device (one per SM),
// with every kernel's shared-memory limit raised once per device.
template <int DT>
cudaError_t resident_ctas(int* out) {
  static std::mutex mu;
  static int cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    e = cudaFuncSetAttribute(stats_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRingBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(residual_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kRingBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(search_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kDecideWarps * kSlotBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stats_kernel<DT>, kThreads,
                                                      kRingBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cache[dev] = per_sm * sms;
  }
  *out = cache[dev];
  return cudaSuccess;
}

cudaError_t resident_ctas_for(specv_dtype dtype, int* out) {
  return dtype == SPECV_BF16 ? resident_ctas<SPECV_BF16>(out) : resident_ctas<SPECV_F32>(out);
}

// CTAs of the stats kernel: enough agents for two chunks each, at most the
// resident count.
int grid_for(int B, int K, int V, specv_dtype dtype, int ctas) {
  const long long items = static_cast<long long>(launch_batch(B)) * (2 * K + 1) *
                          chunks_per_row(V, dtype, kChunkBytes);
  long long want = (items + 2 * kAgents - 1) / (2 * kAgents);
  if (want < 1) want = 1;
  return static_cast<int>(want < ctas ? want : ctas);
}

// Launches kernel<<<grid, block, smem, stream>>>(P) as a programmatic
// dependent of the previous kernel on the stream.
template <class Kern>
cudaError_t launch_dependent(Kern kernel, int grid, int block, int smem, cudaStream_t stream,
                             const Params& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

template <int DT>
cudaError_t launch_sequence(const Params& P, int grid, bool decide_only, cudaStream_t stream) {
  cudaError_t e = launch_dependent(stats_kernel<DT>, grid, kThreads, kRingBytes, stream, P);
  if (e != cudaSuccess) return e;
  const bool walk = P.mode == kModeSample || P.mode == kModeOnehot;
  e = walk ? launch_dependent(decide_kernel<DT, true>, P.B, kDecideWarps * 32, 0, stream, P)
           : launch_dependent(decide_kernel<DT, false>, P.B, kDecideWarps * 32, 0, stream, P);
  if (e != cudaSuccess || decide_only || walk) return e;   // greedy trees list no draws
  e = launch_dependent(residual_kernel<DT>, grid, kThreads, kRingBytes, stream, P);
  // only the verification rule with draft logits lists residual draws (the
  // sampler and the one-hot rule list walks alone)
  if (e != cudaSuccess || P.mode != kModeVerify) return e;
  return launch_dependent(search_kernel<DT>, (P.B + kDecideWarps - 1) / kDecideWarps,
                          kDecideWarps * 32, kDecideWarps * kSlotBytes, stream, P);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The device-visible address of page-locked host memory at p (registered
// or allocated through CUDA), or null for pageable memory and anything
// else: only such an address is ever read by a kernel.
const void* mapped_host(const void* p) {
  cudaPointerAttributes a = {};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();   // pageable memory may report an error on older runtimes
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  return a.devicePointer;
}

uintptr_t up16(uintptr_t x) { return (x + 15) & ~static_cast<uintptr_t>(15); }
uintptr_t down16(uintptr_t x) { return x & ~static_cast<uintptr_t>(15); }

// Everything one call of the library's sampling entry points passes down:
// the verification rule and its variants share the launch sequence.
struct Call {
  int mode = kModeVerify;
  const void* target = nullptr;
  const void* draft = nullptr;
  specv_dtype dtype = SPECV_F32;
  const int32_t* draft_tokens = nullptr;   // tree mode: node tokens [B][K+1]
  const int32_t* draft_len = nullptr;      // tree mode: node counts [B]
  const int32_t* parents = nullptr;        // tree mode
  const float* temperature = nullptr;
  const float* uniforms = nullptr;
  const float* uniforms_resample = nullptr;
  int B = 0, K = 0, V = 0;
  int32_t* accepted_len = nullptr;
  int32_t* out_tokens = nullptr;
  int32_t* path_nodes = nullptr;           // tree mode
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
  float* row_stats = nullptr;
};

bool ok4(const void* p) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % 4 == 0; }

specv_status launch_call(const Call& c, cudaStream_t stream) {
  const int mode = c.mode;
  const int B = c.B, K = c.K, V = c.V;
  const specv_dtype dtype = c.dtype;
  const bool tree = mode == kModeTree, sample = mode == kModeSample;
  // required pointers per mode
  if (!c.target || !c.out_tokens || !c.workspace) return SPECV_ERR_INVALID_ARG;
  if (!sample && (!c.draft_tokens || !c.accepted_len)) return SPECV_ERR_INVALID_ARG;
  if (!tree && (!c.temperature || !c.uniforms)) return SPECV_ERR_INVALID_ARG;
  if ((mode == kModeVerify || mode == kModeOnehot) && !c.uniforms_resample)
    return SPECV_ERR_INVALID_ARG;
  if (tree && (!c.parents || !c.draft_len || !c.path_nodes)) return SPECV_ERR_INVALID_ARG;
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (B < 1 || K < (sample || tree ? 0 : 1) || V < 1) return SPECV_ERR_INVALID_ARG;
  if (B > SPECV_MAX_BATCH || K > (tree ? kMaxTreeNodes - 1 : SPECV_MAX_DRAFT) ||
      V > specv_max_vocab(dtype))
    return SPECV_ERR_UNSUPPORTED;
  const size_t eb = static_cast<size_t>(elt_bytes(dtype));
  if (!aligned(c.target, eb) || (c.draft && !aligned(c.draft, eb)) || !ok4(c.draft_tokens) ||
      !ok4(c.draft_len) || !ok4(c.parents) || !ok4(c.temperature) || !ok4(c.uniforms) ||
      !ok4(c.uniforms_resample) || !ok4(c.accepted_len) || !ok4(c.out_tokens) ||
      !ok4(c.path_nodes) || !aligned(c.workspace, 256) || !ok4(c.row_stats))
    return SPECV_ERR_INVALID_ARG;
  if (c.workspace_bytes < ws_layout(B, K, V, dtype).total) return SPECV_ERR_WORKSPACE;
  const void* target = c.target;
  const void* draft = mode == kModeVerify ? c.draft : nullptr;
  const int32_t* draft_tokens = c.draft_tokens;
  const int32_t* draft_len = c.draft_len;
  const float* temperature = c.temperature;
  const float* uniforms = c.uniforms;
  const float* uniforms_resample = c.uniforms_resample;
  int32_t* accepted_len = c.accepted_len;
  int32_t* out_tokens = c.out_tokens;
  void* workspace = c.workspace;
  float* row_stats = c.row_stats;

  int ctas = 0;
  if (resident_ctas_for(dtype, &ctas) != cudaSuccess || ctas < 1) return SPECV_ERR_CUDA;
  const int grid = grid_for(B, K, V, dtype, ctas);

  const Layout L = ws_layout(B, K, V, dtype);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // Batches beyond one launch sequence run as consecutive sequences on
  // `stream`; each leaves the workspace ready for the next.
  for (int b0 = 0; b0 < B; b0 += kPlanMax) {
    const int Bl = B - b0 < kPlanMax ? B - b0 : kPlanMax;
    Params P;
    P.target = static_cast<const unsigned char*>(target) + static_cast<size_t>(b0) * (K + 1) * V * eb;
    P.draft = draft ? static_cast<const unsigned char*>(draft) + static_cast<size_t>(b0) * K * V * eb
                    : nullptr;
    const size_t tok_stride = tree ? static_cast<size_t>(K + 1) : static_cast<size_t>(K);
    P.draft_tokens = draft_tokens ? draft_tokens + static_cast<size_t>(b0) * tok_stride : nullptr;
    P.draft_len = draft_len ? draft_len + b0 : nullptr;
    P.parents = c.parents ? c.parents + static_cast<size_t>(b0) * (K + 1) : nullptr;
    P.temperature = temperature ? temperature + b0 : nullptr;
    P.uniforms = uniforms ? uniforms + static_cast<size_t>(b0) * (K + 1) : nullptr;
    P.uniforms_resample = uniforms_resample ? uniforms_resample + b0 : nullptr;
    P.B = Bl;
    P.K = K;
    P.V = V;
    P.mode = mode;
    P.R = 2 * K + 1;
    P.NC = chunks_per_row(V, dtype, kChunkBytes);
    P.NCd = chunks_per_row(V, dtype, kDrawBytes);
    P.inv_NC = 1.0f / static_cast<float>(P.NC);
    const uintptr_t t0 = reinterpret_cast<uintptr_t>(P.target);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(P.draft);
    P.t_lo = up16(t0);
    P.t_hi = down16(t0 + static_cast<size_t>(Bl) * (K + 1) * V * eb);
    P.d_lo = draft ? up16(d0) : 0;
    P.d_hi = draft ? down16(d0 + static_cast<size_t>(Bl) * K * V * eb) : 0;
    P.accepted_len = accepted_len ? accepted_len + b0 : nullptr;
    P.out_tokens = out_tokens + static_cast<size_t>(b0) * (K + 1);
    P.path_nodes = c.path_nodes ? c.path_nodes + static_cast<size_t>(b0) * (K + 1) : nullptr;
    P.header = reinterpret_cast<int32_t*>(ws + L.header);
    P.req = reinterpret_cast<Req*>(ws + L.req);
    P.part = reinterpret_cast<uint2*>(ws + L.part);
    P.zx = reinterpret_cast<float*>(ws + L.zx);
    P.dpc = reinterpret_cast<float*>(ws + L.dpc);
    P.row_stats = row_stats ? row_stats + static_cast<size_t>(b0) * (K + 1) * 8 : nullptr;
    const cudaError_t e = dtype == SPECV_BF16 ? launch_sequence<SPECV_BF16>(P, grid, tree, stream)
                                              : launch_sequence<SPECV_F32>(P, grid, tree, stream);
    if (e != cudaSuccess) return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

specv_status launch(const void* target, const void* draft, specv_dtype dtype,
                    const int32_t* draft_tokens, const int32_t* draft_len,
                    const float* temperature, const float* uniforms,
                    const float* uniforms_resample, int B, int K, int V, int32_t* accepted_len,
                    int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                    float* row_stats, cudaStream_t stream) {
  Call c;
  c.mode = kModeVerify;
  c.target = target;
  c.draft = draft;
  c.dtype = dtype;
  c.draft_tokens = draft_tokens;
  c.draft_len = draft_len;
  c.temperature = temperature;
  c.uniforms = uniforms;
  c.uniforms_resample = uniforms_resample;
  c.B = B;
  c.K = K;
  c.V = V;
  c.accepted_len = accepted_len;
  c.out_tokens = out_tokens;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.row_stats = row_stats;
  return launch_call(c, stream);
}

size_t pad256(size_t x) { return align256(x); }

// ---------------------------------------------------------------- no-allocation scratch
//
// Scratch for spec_verify_sample_noalloc: the same layout as a caller's
// workspace, at most SPECV_NOALLOC_SCRATCH_BYTES.  It is a module-scope
// device array, so every GPU that loads this library holds it until the
// process exits, and every call on a device shares it.
__device__ __align__(256) unsigned char g_noalloc_scratch[SPECV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current device's context.  In
// host code the symbol's name is only a host-side handle, so the address is
// looked up with cudaGetSymbolAddress, with the device current, on every
// call: a lookup is a host-side table read once the module is loaded, and a
// context that was reset and recreated (cudaDeviceReset) gets its new
// address instead of a stale one.
cudaError_t noalloc_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

// ---------------------------------------------------------------- C ABI

extern "C" {

int specv_version(void) { return 500; }

int specv_max_vocab(specv_dtype dtype) {
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return 0;
  return kMaxRowBytes / elt_bytes(dtype);
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
  return ws_layout(B, K, V, dtype).total;
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
  // Only the rows the kernels read cross the host link (its bandwidth bounds
  // this entry point): a usable request's target rows t <= n_b and, when it
  // samples, its draft rows t < n_b -- the rule the device applies to the
  // same draft_len and temperature.  Page-locked logits with 16-byte rows
  // are gathered by one kernel reading host memory; otherwise each range of
  // adjacent rows goes as one copy.
  bool ok = true;
  const size_t row = static_cast<size_t>(V) * eb;
  const void* ht = mapped_host(target_logits);
  const void* hd = draft_logits ? mapped_host(draft_logits) : nullptr;
  const bool gather = ht && (!draft_logits || hd) && row % 16 == 0 &&
                      aligned(ht, 16) && (!hd || aligned(hd, 16)) && aligned(d_t, 16) &&
                      (!d_d || aligned(d_d, 16));
  if (!gather) {
    size_t t_lo = 0, t_hi = 0, d_lo = 0, d_hi = 0;   // pending ranges (bytes)
    auto flush = [&](void* dst, const void* src, size_t lo, size_t hi) {
      if (hi > lo)
        ok = ok && h2d(static_cast<unsigned char*>(dst) + lo, static_cast<const unsigned char*>(src) + lo,
                       hi - lo);
    };
    for (int b = 0; b < B && ok; ++b) {
      const int n = draft_len ? draft_len[b] : K;
      const float T = temperature[b];
      if (n < 1 || n > K || !(T >= 0.0f) || std::isinf(T)) continue;   // flagged on the device
      const bool sampled = T > 0.0f;
      if (sampled && !draft_logits) continue;
      const size_t t0 = static_cast<size_t>(b) * (K + 1) * row, t1 = t0 + static_cast<size_t>(n + 1) * row;
      if (t0 != t_hi) {
        flush(d_t, target_logits, t_lo, t_hi);
        t_lo = t0;
      }
      t_hi = t1;
      if (sampled) {
        const size_t q0 = static_cast<size_t>(b) * K * row, q1 = q0 + static_cast<size_t>(n) * row;
        if (q0 != d_hi) {
          flush(d_d, draft_logits, d_lo, d_hi);
          d_lo = q0;
        }
        d_hi = q1;
      }
    }
    flush(d_t, target_logits, t_lo, t_hi);
    if (draft_logits) flush(d_d, draft_logits, d_lo, d_hi);
  }
  ok = ok && h2d(d_tok, draft_tokens, static_cast<size_t>(B) * K * 4);
  if (draft_len) ok = ok && h2d(d_len, draft_len, static_cast<size_t>(B) * 4);
  ok = ok && h2d(d_T, temperature, static_cast<size_t>(B) * 4);
  ok = ok && h2d(d_u, uniforms, static_cast<size_t>(B) * (K + 1) * 4);
  ok = ok && h2d(d_ur, uniforms_resample, static_cast<size_t>(B) * 4);
  if (!ok) return SPECV_ERR_CUDA;
  if (gather) {
    int ctas = 0;
    if (resident_ctas_for(dtype, &ctas) != cudaSuccess || ctas < 1) return SPECV_ERR_CUDA;
    const long long slots = static_cast<long long>(B) * (2 * K + 1);
    const int grid = static_cast<int>(std::min<long long>(slots, 4LL * ctas));
    gather_rows_kernel<<<grid, kGatherThreads, 0, s>>>(
        static_cast<const uint4*>(ht), static_cast<const uint4*>(hd), static_cast<uint4*>(d_t),
        static_cast<uint4*>(d_d), draft_len ? d_len : nullptr, d_T, B, K, row / 16);
    if (cudaGetLastError() != cudaSuccess) return SPECV_ERR_CUDA;
  }
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
  int ctas = 0;
  if (resident_ctas_for(dtype, &ctas) != cudaSuccess) return SPECV_ERR_CUDA;
  out[0] = grid_for(B, K, V, dtype, ctas);
  out[1] = kChunkBytes / elt_bytes(dtype);
  out[2] = kSlots;
  out[3] = chunks_per_row(V, dtype, kChunkBytes);
  out[4] = kRingBytes;
  out[5] = kThreads;
  return SPECV_OK;
}

size_t specv_sample_workspace_bytes(int R, int V, specv_dtype dtype) {
  if (R < 1 || V < 1 || R > SPECV_MAX_BATCH || (dtype != SPECV_F32 && dtype != SPECV_BF16) ||
      V > specv_max_vocab(dtype))
    return 0;
  return ws_layout(R, 0, V, dtype).total;
}

specv_status spec_sample_draft(const void* logits, specv_dtype dtype, const float* temperature,
                               const float* uniforms, int R, int V, int32_t* tokens,
                               void* workspace, size_t workspace_bytes, float* row_stats,
                               specv_stream_t stream) {
  Call c;
  c.mode = kModeSample;
  c.target = logits;
  c.dtype = dtype;
  c.temperature = temperature;
  c.uniforms = uniforms;
  c.B = R;
  c.K = 0;
  c.V = V;
  c.out_tokens = tokens;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.row_stats = row_stats;
  return launch_call(c, reinterpret_cast<cudaStream_t>(stream));
}

specv_status spec_verify_sample_onehot(const void* target_logits, specv_dtype dtype,
                                       const int32_t* draft_tokens, const int32_t* draft_len,
                                       const float* temperature, const float* uniforms,
                                       const float* uniforms_resample, int B, int K, int V,
                                       int32_t* accepted_len, int32_t* out_tokens,
                                       void* workspace, size_t workspace_bytes,
                                       float* row_stats, specv_stream_t stream) {
  Call c;
  c.mode = kModeOnehot;
  c.target = target_logits;
  c.dtype = dtype;
  c.draft_tokens = draft_tokens;
  c.draft_len = draft_len;
  c.temperature = temperature;
  c.uniforms = uniforms;
  c.uniforms_resample = uniforms_resample;
  c.B = B;
  c.K = K;
  c.V = V;
  c.accepted_len = accepted_len;
  c.out_tokens = out_tokens;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.row_stats = row_stats;
  return launch_call(c, reinterpret_cast<cudaStream_t>(stream));
}

size_t specv_tree_workspace_bytes(int B, int N, int V, specv_dtype dtype) {
  if (B < 1 || N < 1 || V < 1 || B > SPECV_MAX_BATCH || N > kMaxTreeNodes ||
      (dtype != SPECV_F32 && dtype != SPECV_BF16) || V > specv_max_vocab(dtype))
    return 0;
  return ws_layout(B, N - 1, V, dtype).total;
}

specv_status spec_verify_tree_greedy(const void* target_logits, specv_dtype dtype,
                                     const int32_t* parents, const int32_t* tokens,
                                     const int32_t* n_nodes, int B, int N, int V,
                                     int32_t* accepted_len, int32_t* out_tokens,
                                     int32_t* path_nodes, void* workspace,
                                     size_t workspace_bytes, float* row_stats,
                                     specv_stream_t stream) {
  if (N < 1) return SPECV_ERR_INVALID_ARG;
  Call c;
  c.mode = kModeTree;
  c.target = target_logits;
  c.dtype = dtype;
  c.draft_tokens = tokens;
  c.draft_len = n_nodes;
  c.parents = parents;
  c.B = B;
  c.K = N - 1;
  c.V = V;
  c.accepted_len = accepted_len;
  c.out_tokens = out_tokens;
  c.path_nodes = path_nodes;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.row_stats = row_stats;
  return launch_call(c, reinterpret_cast<cudaStream_t>(stream));
}

specv_status spec_insert_accepted(const int32_t* accepted_len, const int32_t* out_tokens, int B,
                                  int K, int32_t* seq_lens, int32_t* history, int L,
                                  int32_t* next_tokens, int32_t* cu_emitted, int32_t* packed,
                                  int32_t* status, specv_stream_t stream) {
  if (!accepted_len || !out_tokens || !seq_lens || !history || !next_tokens || !cu_emitted ||
      !packed || !status)
    return SPECV_ERR_INVALID_ARG;
  if (B < 1 || K < 0 || L < 1) return SPECV_ERR_INVALID_ARG;
  if (B > SPECV_MAX_BATCH || K > kMaxTreeNodes) return SPECV_ERR_UNSUPPORTED;
  if (!ok4(accepted_len) || !ok4(out_tokens) || !ok4(seq_lens) || !ok4(history) ||
      !ok4(next_tokens) || !ok4(cu_emitted) || !ok4(packed) || !ok4(status))
    return SPECV_ERR_INVALID_ARG;
  insert_kernel<<<1, kInsertThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      accepted_len, out_tokens, B, K + 1, seq_lens, history, L, next_tokens, cu_emitted, packed,
      status);
  return cudaGetLastError() == cudaSuccess ? SPECV_OK : SPECV_ERR_CUDA;
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
