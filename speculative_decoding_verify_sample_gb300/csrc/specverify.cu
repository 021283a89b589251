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
// Design.  Every warp of the grid is an independent agent.  The logits a
// call needs are cut into items of one 8 KB chunk of one row ("stats"
// items), numbered request by request, and agent a takes items a, a + G,
// a + 2G, ... (G agents).  An agent streams its items through a private ring
// of three shared-memory slots with TMA bulk copies, each slot completing on
// its own mbarrier, and reduces each chunk alone to a partial: the chunk's
// maximum and sum of exp((z - max)/T), or at T = 0 its maximum and the
// lowest index holding it.  It then counts the item on the request's
// counter in global memory.  The agent whose count completes a request
// combines the request's partials, runs the left-to-right accept test and
// either answers the request (greedy, or bad data) or publishes the final
// row for the draw.  The final row (the residual (p - q)+ at a rejected
// position, p at the bonus position) is read again as "draw" items of 4 KB
// of target and draft each; draw item d of the request-major draw space
// belongs to agent d mod G, which polls the request's state between its
// stats items.  A draw item stores per-sweep sums of the final-draw weights;
// the agent whose count completes the draw locates the token from them,
// re-reading one 512-byte segment, and writes the outputs.
//
// No agent waits on another while it still has stats items: a wait for a
// decision happens only once its own ring is empty and its counts are
// flushed, so every wait ends.  Every wait is also bounded in time and sets
// a status bit when it gives up.  Each needed logit is read from HBM once;
// the final row of a sampled request is read a second time, normally from
// L2, because items run request by request.

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

constexpr int kAgents = 8;                              // agent warps per CTA
constexpr int kThreads = (kAgents + 1) * 32;            // + the control warp
constexpr int kSlots = 2;                               // ring slots per agent
constexpr int kChunkBytes = 12288;                      // stats item: one chunk of one row
constexpr int kDrawBytes = 4096;                        // draw item: this much of the target row
constexpr int kDrawSweeps = kDrawBytes / 512;           // 32 lanes x 16 bytes per sweep
constexpr int kDraftOff = kDrawBytes;                   // draft part of a draw slot
constexpr int kSlotBytes = kChunkBytes + 32;            // >= kDraftOff + kDrawBytes + 16
constexpr int kMassMax = 520;                           // chunks per row, either size
constexpr int kRingBytes = kAgents * kSlots * kSlotBytes;
constexpr int kCtlRecords = 2080;                       // control-warp staging (8-byte records)
constexpr int kPend = 16;                               // decided requests awaiting their draw
constexpr int kMaxRowBytes = 1 << 21;                   // 2 MB per row of logits
constexpr long long kWaitLimitCycles = 4000000000ll;    // ~2 s at 2 GHz
constexpr uint32_t kSuspendHintNs = 20000;

static_assert(kSlotBytes >= kDraftOff + kDrawBytes + 16, "draw slot too small");
static_assert(kSlotBytes % 16 == 0, "slots must keep 16-byte alignment");
static_assert(kDrawSweeps == 8, "a draw chunk has eight sweeps");
static_assert(kCtlRecords >= 513, "the draw records of a 2 MB row fit the staging buffer");
static_assert(kCtlRecords * 8 >= kChunkBytes + 16 && kCtlRecords * 8 >= kDraftOff + kDrawBytes + 16,
              "a chunk of logits fits the control warp's buffer");
static_assert(kMassMax >= (kMaxRowBytes + 15) / kDrawBytes + 1, "chunk masses of a 2 MB row fit");

// workspace header words, one 128-byte line each
constexpr int kHStatus = 0, kHExit = 32, kHEpoch = 64;
constexpr int kHeaderBytes = 512;

// per-request decision state: (call tag << 32) | payload, payload =
// kind | residual << 2 | final row << 3
constexpr uint32_t kStateDraws = 1, kStateNone = 2;

// A record is one 8-byte word written at once; bit 31 of its high half is
// set in every written record, so a zero record is "not written yet".
constexpr uint32_t kReady = 0x80000000u;

constexpr int kItemStats = 1, kItemDraw = 2;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Per-request record in the workspace (64 bytes).
struct __align__(16) Req {
  unsigned long long state;   // decision, tagged with the call
  int pad0[6];
  float4 prm;                 // final row: Mp, Mq, log2(e)/T, S_p/S_q
  float pad1[4];
};
static_assert(sizeof(Req) == 64, "Req is one 64-byte record");

struct Params {
  const unsigned char* target;
  const unsigned char* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  const float* uniforms;
  const float* uniforms_resample;
  int B, K, V;
  int R;            // record rows per request: K+1 target, then K draft
  int NC;           // stats chunks per row
  int NCd;          // draw chunks per row
  float inv_NC;     // 1 / NC
  // 16-byte-aligned address ranges the bulk copies may read
  uintptr_t t_lo, t_hi, d_lo, d_hi;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t* header;
  Req* req;         // [B]
  uint2* part;      // [B][R][NC] stats records: (max, sum | ready) or (max, index | ready)
  uint2* dpart;     // [B][NCd] draw records: (0, residual mass | ready)
  uint2* zx;        // [B][R] records of the drafted token's logit in rows t < n: (z, ready)
  float* row_stats; // [B][K+1][8] or null
};

// One item as its agent staged it (48 bytes).
struct __align__(16) Item {
  int kind;     // kItemStats / kItemDraw
  int b;
  int row;      // stats: t (target) or K+1+t (draft); draw: final row t
  int c;        // chunk
  int mode;     // stats: greedy; draw: residual
  float sT;     // stats: log2(e)/T
  int xrow;     // stats: t if the row's drafted token x_t is needed, else -1
  int peek_b;   // request whose state `peek` samples (-1: none)
  // copied in with the slot (cp.async on the slot's barrier):
  unsigned long long peek;   // state of request peek_b when the item was staged
  unsigned long long peek_pad;
  int x;                     // x_t (when xrow >= 0)
  int pad[3];
  float4 prm;   // draw: the decision's Mp, Mq, log2(e)/T, S_p/S_q
};

struct AgentSmem {
  uint64_t full[kSlots];
  Item item[kSlots];
};

// A decided request whose final draw is pending (the control warp's).
struct __align__(16) Pend {
  int b, j, t_f, residual;
  float u, Sp, pad0, pad1;
  float4 prm;
};

struct Smem {
  AgentSmem ag[kAgents];
  alignas(128) uint2 cbuf[kCtlRecords];   // control warp: staged records, or a chunk of logits
  uint64_t cbar;                          // control warp: its chunk copies
  float cmass[kMassMax];     // control warp: chunk masses of a final draw
  Pend pend[kPend];
  uint32_t tag;
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

// Non-tensor TMA bulk copy global -> this CTA's shared memory.  Both
// addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, uintptr_t src, uint32_t bytes,
                                              uint64_t* bar) {
  const unsigned long long gsrc =
      static_cast<unsigned long long>(__cvta_generic_to_global(reinterpret_cast<const void*>(src)));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(__cvta_generic_to_global(p)));
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
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

__device__ __forceinline__ int request_bad(const Params& P, int n, float T) {
  if (n < 1 || n > P.K) return SPECV_DEV_BAD_DRAFT_LEN;
  if (!(T >= 0.0f) || isinf(T)) return SPECV_DEV_BAD_TEMPERATURE;
  if (T > 0.0f && P.draft == nullptr) return SPECV_DEV_NO_DRAFT;
  return 0;
}

// Stats items of a request: target rows t <= n, draft rows t < n when
// sampled, every chunk; none if its length or temperature is unusable.
__device__ __forceinline__ int request_items(const Params& P, int n, float T) {
  if (request_bad(P, n, T)) return 0;
  return ((n + 1) + (T > 0.0f ? n : 0)) * P.NC;
}

__device__ __forceinline__ int request_len(const Params& P, int b) {
  return P.draft_len ? __ldg(P.draft_len + b) : P.K;
}

// Whole warp: writes a request's outputs.
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
  if (lane == 0) P.accepted_len[b] = j;
  __syncwarp();
}

// Publishes request b's decision for the agents that own its draw items.
__device__ __forceinline__ void set_state(const Params& P, int b, uint32_t tag, uint32_t payload) {
  cuda::atomic_ref<unsigned long long, cuda::thread_scope_device>(P.req[b].state)
      .store((static_cast<unsigned long long>(tag) << 32) | payload, cuda::memory_order_release);
}

__device__ void finish_bad(const Params& P, int b, int bits, int lane, uint32_t tag) {
  if (lane == 0) {
    atomicOr(P.header + kHStatus, bits);
    set_state(P, b, tag, kStateNone);
  }
  finish_request(P, b, -1, -1, lane);
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
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 2
  for (int j = vs.vf0 + lane; j < vs.vf1; j += 32) {
    float v[CH];
    E::unpack(vec[j], v);
#pragma unroll
    for (int q = 0; q < CH; q += 2) {
      s0 = __fadd_rn(s0, ex2(__fmaf_rn(v[q], sT, -c)));
      s1 = __fadd_rn(s1, ex2(__fmaf_rn(v[q + 1], sT, -c)));
    }
  }
  if (my_edge >= 0) {
#pragma unroll
    for (int q = 0; q < CH; ++q) s0 = __fadd_rn(s0, ex2(__fmaf_rn(ev[q], sT, -c)));
  }
  const float S = warp_sum(__fadd_rn(s0, s1));
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
#pragma unroll
  for (int q = 0; q < CH; ++q) w[q] = weight(vp[q], vq[q], residual, prm);
}

// Whole warp: the final-draw mass of a draw chunk: per sweep of 32 vectors
// (sweep s = vectors [32 s, 32 s + 32) of the target part) each lane's
// elements in order, then across the warp, then the sweeps in order (as
// draw_in_slot walks them).
template <int DT>
__device__ __forceinline__ float chunk_draw(const unsigned char* slot, const Chunk& kp,
                                            const Chunk& kq, bool residual, const float4& prm,
                                            int lane) {
  constexpr int CH = Elt<DT>::kPerVec;
  const Vecs vs = vecs_of<DT>(kp);
  const bool same = kq.off0 == kp.off0;   // draft elements at the target's positions
  float t = 0.0f;
#pragma unroll 1
  for (int s = 0; s < kDrawSweeps; ++s) {
    float w[CH];
    vector_weights<DT>(slot, vs, kp, kq, residual, same, prm, s * 32 + lane, w);
    float s0 = 0.0f;
#pragma unroll
    for (int q = 0; q < CH; ++q) s0 = __fadd_rn(s0, w[q]);
    t = __fadd_rn(t, warp_sum(s0));
  }
  return t;
}

// Whole warp: the final draw's token inside a chunk staged in a slot.
// `tau` is the target mass left for this chunk; sweeps (32 vectors each)
// are summed in order as chunk_draw sums them, then lanes in order, then
// the lane's elements.  Rounding that leaves tau beyond the chunk's mass
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

// ---------------------------------------------------------------- records

__device__ __forceinline__ void st_record(uint2* p, uint32_t lo, uint32_t hi) {
  const unsigned long long v = (static_cast<unsigned long long>(hi) << 32) | lo;
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint2 ld_record(const uint2* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return make_uint2(static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32));
}

// A nonnegative (or NaN) float with the ready bit, and back.
__device__ __forceinline__ uint32_t ready_bits(float x) {
  return (x != x ? 0x7FC00000u : __float_as_uint(x)) | kReady;
}
__device__ __forceinline__ float ready_value(uint32_t u) { return __uint_as_float(u & ~kReady); }

// Whole warp: stages n records from src into dst, up to 16 loads in flight
// per lane; true if every one of them is written.
__device__ __forceinline__ bool stage_records(uint2* dst, const uint2* src, int n, int lane) {
  bool ready = true;
  for (int base = 0; base < n; base += 16 * 32) {
    uint2 v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int i = base + k * 32 + lane;
      if (i < n) v[k] = ld_record(src + i);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int i = base + k * 32 + lane;
      if (i < n) {
        dst[i] = v[k];
        ready = ready && (v[k].y & kReady);
      }
    }
  }
  return __all_sync(0xffffffffu, ready);
}

// Whole warp: returns n records to "not written" for the next call.
__device__ __forceinline__ void clear_records(uint2* p, int n, int lane) {
  for (int i = lane; i < n; i += 32) p[i] = make_uint2(0u, 0u);
}

// ---------------------------------------------------------------- decisions

// (max, sum) of one row from its NC staged stats records: the maximum
// first, then the chunk sums rescaled to it, in chunk order.
__device__ __forceinline__ void combine_row(const uint2* p, int NC, float sT, float& M, float& S) {
  M = -INFINITY;
  for (int c = 0; c < NC; ++c) M = fmaxf(M, __uint_as_float(p[c].x));
  S = 0.0f;
  if (M == -INFINITY) return;
  for (int c = 0; c < NC; ++c) {
    const float m = __uint_as_float(p[c].x);
    if (m > -INFINITY) S = __fadd_rn(S, __fmul_rn(ready_value(p[c].y), scaled_exp(m, M, sT)));
  }
}

// Argmax of one row from its staged records: chunks are in index order, so
// the first chunk holding the maximum has the lowest index.
__device__ __forceinline__ void argmax_row(const uint2* p, int NC, float& v, int& i) {
  v = __uint_as_float(p[0].x);
  i = static_cast<int>(p[0].y & ~kReady);
  for (int c = 1; c < NC; ++c) {
    const float m = __uint_as_float(p[c].x);
    if (m > v) {
      v = m;
      i = static_cast<int>(p[c].y & ~kReady);
    }
  }
}

// Whole warp: stages request b's records of target rows [0, nt) and draft
// rows [0, nd) pass by pass and combines them: lane t gets target row t
// (Mp, Sp, or the argmax) and draft row t (Mq, Sq).  False if a record is
// not written yet.
__device__ bool combine_request(const Params& P, Smem& S, int b, int nt, int nd, bool greedy,
                                float sT, int lane, float& Mp, float& Sp, float& Mq, float& Sq,
                                int& arg) {
  const int NC = P.NC, K = P.K;
  uint2* buf = S.cbuf;
  const int cap = max(1, kCtlRecords / NC);   // rows per pass
  const uint2* rec = P.part + static_cast<size_t>(b) * P.R * NC;
  Mp = Mq = -INFINITY;
  Sp = Sq = 0.0f;
  arg = INT_MAX;
  for (int v0 = 0; v0 < nt + nd; v0 += cap) {
    const int v1 = min(nt + nd, v0 + cap);
    // virtual rows [v0, v1): target rows first, then draft rows
    const int ta = v0, tb = min(v1, nt);
    const int da = max(v0, nt) - nt, db = v1 - nt;
    const int ntr = max(0, tb - ta);
    bool ready = true;
    if (ntr > 0) ready = stage_records(buf, rec + static_cast<size_t>(ta) * NC, ntr * NC, lane);
    if (db > da)
      ready = stage_records(buf + ntr * NC, rec + static_cast<size_t>(K + 1 + da) * NC,
                            (db - da) * NC, lane) && ready;
    __syncwarp();
    if (!ready) return false;
    if (lane >= ta && lane < tb) {
      const uint2* p = buf + (lane - ta) * NC;
      if (greedy) argmax_row(p, NC, Mp, arg);
      else combine_row(p, NC, sT, Mp, Sp);
    }
    if (lane >= da && lane < db) combine_row(buf + (ntr + lane - da) * NC, NC, sT, Mq, Sq);
    __syncwarp();
  }
  return true;
}

// Whole warp: the chunk holding mass u * W of a draw, chunk masses
// mass[0..n) in shared memory (lane l sums chunks [l m, l m + m) in order,
// then the lanes are scanned).  Returns the chunk and, in rem, the target
// mass left inside it; rounding that leaves the target beyond the total
// falls on the last chunk with positive mass.  Sets W to the total.  -1:
// no mass at all.
__device__ int pick_chunk(const float* mass, int n, float u, int lane, float& W, float& rem) {
  const int m = (n + 31) / 32;
  const int c0 = min(n, lane * m), c1 = min(n, c0 + m);
  float lane_tot = 0.0f;
  for (int c = c0; c < c1; ++c) lane_tot = __fadd_rn(lane_tot, mass[c]);
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
      const float t = mass[c];
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
template <int DT>
__device__ bool ctl_fetch(const Params& P, Smem& S, uint32_t& cphase, uintptr_t rp, uintptr_t rq,
                          int c, int CB, bool residual, Chunk& kp, Chunk& kq, int lane) {
  unsigned char* slot = reinterpret_cast<unsigned char*>(S.cbuf);
  kp = chunk_of<DT>(rp, P.V, c, CB);
  kq = residual ? draft_part<DT>(rq, kp) : kp;
  __syncwarp();   // every lane is done with the buffer
  if (lane == 0) {
    uintptr_t s0 = 0, s1 = 0;
    const uint32_t n0 = bulk_span<DT>(kp, P.t_lo, P.t_hi, &s0);
    const uint32_t n1 = residual ? bulk_span<DT>(kq, P.d_lo, P.d_hi, &s1) : 0u;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&S.cbar, n0 + n1);
    if (n0) bulk_copy_g2s(slot + (s0 - kp.g0), s0, n0, &S.cbar);
    if (n1) bulk_copy_g2s(slot + kDraftOff + (s1 - kq.g0), s1, n1, &S.cbar);
  }
  const bool ok = warp_wait(&S.cbar, cphase & 1u);
  ++cphase;
  if (!ok && lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
  fix_edges<DT>(kp, P.t_lo, P.t_hi, slot, lane);
  if (residual) fix_edges<DT>(kq, P.d_lo, P.d_hi, slot + kDraftOff, lane);
  return ok;
}

// Whole warp: out_tokens[b] = x_0 .. x_{j-1}, tok at j (skipped if
// skip_j), -1 after; accepted_len[b] = j.  Lane s < n holds x_s.
__device__ __forceinline__ void write_outputs(const Params& P, int b, int j, int tok, int x_lane,
                                              bool skip_j, int lane) {
  if (lane <= P.K && !(skip_j && lane == j))
    P.out_tokens[static_cast<size_t>(b) * (P.K + 1) + lane] = lane < j ? x_lane : (lane == j ? tok : -1);
  if (lane == 0) P.accepted_len[b] = j;
}

// Whole warp (control): tries to decide request b.  Returns 0 if some of
// its records are not written yet, 1 if the request is answered (greedy, a
// bonus draw, or bad data), 2 if its rejected row is published for the
// residual draw (pe filled, every output but the drawn token written).
// Validates the request's tokens and uniforms, combines its records, runs
// the rule's left-to-right test; a bonus draw (every draft accepted) is
// taken at once from the final row's chunk masses, which its records give,
// and one re-read chunk.
template <int DT>
__device__ __noinline__ int try_decide(const Params& P, Smem& S, uint32_t& cphase, int b, int n,
                                       float T, int lane, uint32_t tag, Pend& pe) {
  const int K = P.K, V = P.V, NC = P.NC, R = P.R;
  const bool greedy = !(T > 0.0f);
  const int nt = n + 1, nd = greedy ? 0 : n;
  uint2* rec = P.part + static_cast<size_t>(b) * R * NC;
  uint2* zrec = P.zx + static_cast<size_t>(b) * R;
  int x_lane = -1;
  float u_lane = 0.0f;
  if (lane < n) x_lane = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + lane);
  if (lane <= n) u_lane = __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + lane);
  const float ur = __ldg(P.uniforms_resample + b);
  // the drafted tokens' logits (sampled rows t < n)
  uint2 zp_r = make_uint2(0u, kReady), zq_r = make_uint2(0u, kReady);
  if (!greedy && lane < n) {
    zp_r = ld_record(zrec + lane);
    zq_r = ld_record(zrec + K + 1 + lane);
  }
  const float sT = greedy ? 0.0f : temp_scale(T);
  float Mp_l, Sp_l, Mq_l, Sq_l;
  int g;
  if (!combine_request(P, S, b, nt, nd, greedy, sT, lane, Mp_l, Sp_l, Mq_l, Sq_l, g)) return 0;
  const bool tok_bad = lane < n && (x_lane < 0 || x_lane >= V);
  const bool u_bad = lane <= n && !(u_lane >= 0.0f && u_lane < 1.0f);
  int bad = 0;
  if (__any_sync(0xffffffffu, tok_bad)) bad |= SPECV_DEV_BAD_TOKEN;
  if (__any_sync(0xffffffffu, u_bad) || !(ur >= 0.0f && ur < 1.0f)) bad |= SPECV_DEV_BAD_UNIFORM;
  // a valid token's logit record is written by the item holding it
  if (!bad && !__all_sync(0xffffffffu, (zp_r.y & kReady) && (zq_r.y & kReady))) return 0;

  float* rs = P.row_stats ? P.row_stats + static_cast<size_t>(b) * (K + 1) * 8 : nullptr;
  int result = 1;
  if (bad) {
    finish_bad(P, b, bad, lane, tag);
  } else if (greedy) {
    if (rs && lane <= n) {
      rs[lane * 8 + 0] = Mp_l;
      rs[lane * 8 + 7] = static_cast<float>(g);
    }
    const unsigned miss = __ballot_sync(0xffffffffu, lane < n && g != x_lane);
    const int j = miss ? __ffs(miss) - 1 : n;
    const int gj = __shfl_sync(0xffffffffu, g, j);
    if (gj < 0 || gj >= V) {
      finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, tag);
    } else {
      if (lane == 0) set_state(P, b, tag, kStateNone);
      write_outputs(P, b, j, gj, x_lane, false, lane);
    }
  } else {
    // ---- sampled: lane t holds target row t and draft row t ----------------
    const bool row_bad = (lane <= n && !isfinite(Mp_l)) || (lane < n && !isfinite(Mq_l));
    if (__any_sync(0xffffffffu, row_bad)) {
      finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, tag);
    } else {
      float lp = 0.0f, lq = 0.0f;
      if (lane < n) {
        lp = __fsub_rn(__fmul_rn(__fsub_rn(__uint_as_float(zp_r.x), Mp_l), sT), log2f(Sp_l));
        lq = __fsub_rn(__fmul_rn(__fsub_rn(__uint_as_float(zq_r.x), Mq_l), sT), log2f(Sq_l));
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
      if (j == n) {
        // bonus draw from p_n: chunk masses s_c 2^((m_c - Mp) log2(e)/T)
        const uint2* rn = rec + static_cast<size_t>(n) * NC;
        for (int c = lane; c < NC; c += 32) {
          const uint2 r = ld_record(rn + c);
          const float m = __uint_as_float(r.x);
          S.cmass[c] = m > -INFINITY ? __fmul_rn(ready_value(r.y), scaled_exp(m, Mp, sT)) : 0.0f;
        }
        __syncwarp();
        float W, rem;
        const int chunk = pick_chunk(S.cmass, NC, u_bonus, lane, W, rem);
        const float4 prm = make_float4(Mp, 0.0f, sT, 0.0f);
        const uintptr_t rp = row_addr<DT>(P.target, static_cast<size_t>(b) * (K + 1) + n, V);
        int tok = -1;
        if (chunk >= 0) {
          Chunk kp, kq;
          if (ctl_fetch<DT>(P, S, cphase, rp, 0, chunk, kChunkBytes, false, kp, kq, lane))
            tok = draw_in_slot<DT>(reinterpret_cast<const unsigned char*>(S.cbuf), kp, kq, false,
                                   prm, rem, kChunkBytes / 512, lane);
        }
        if (rs && lane == 0) {
          rs[n * 8 + 6] = __fdiv_rn(W, Sp);
          rs[n * 8 + 7] = static_cast<float>(tok);
        }
        if (tok < 0 || tok >= V) {
          finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, tag);
        } else {
          if (lane == 0) set_state(P, b, tag, kStateNone);
          write_outputs(P, b, n, tok, x_lane, false, lane);
        }
      } else {
        pe.b = b;
        pe.j = j;
        pe.t_f = j;
        pe.residual = 1;
        pe.u = ur;
        pe.Sp = Sp;
        pe.pad0 = pe.pad1 = 0.0f;
        pe.prm = make_float4(Mp, Mq, sT, __fdiv_rn(Sp, Sq));
        write_outputs(P, b, j, -1, x_lane, true, lane);
        if (lane == 0) {
          P.req[b].prm = pe.prm;
          set_state(P, b, tag, kStateDraws | 4u | (static_cast<uint32_t>(j) << 3));
        }
        result = 2;
      }
    }
  }
  // every record of the request is consumed: clear them for the next call
  // (a residual draw keeps its target row's, for the search's fallback to p)
  __syncwarp();
  if (result == 2) {
    clear_records(rec, pe.t_f * NC, lane);
    clear_records(rec + static_cast<size_t>(pe.t_f + 1) * NC, (nt - pe.t_f - 1) * NC, lane);
  } else {
    clear_records(rec, nt * NC, lane);
  }
  if (nd) clear_records(rec + static_cast<size_t>(K + 1) * NC, nd * NC, lane);
  if (!greedy && lane < n) {
    zrec[lane] = make_uint2(0u, 0u);
    zrec[K + 1 + lane] = make_uint2(0u, 0u);
  }
  __syncwarp();
  return result;
}

// Whole warp (control): tries to draw the final token of a request whose
// rejected row is published.  Returns false if some of its draw records
// are not written yet.  Picks the chunk from the records' residual masses
// and searches it, re-read; a residual of exactly zero mass falls back to
// drawing from p with the same uniform, its chunk masses taken from the
// row's stats records (kept for this) and a stats-sized chunk re-read.
template <int DT>
__device__ __noinline__ bool try_search(const Params& P, Smem& S, uint32_t& cphase, const Pend& pe,
                                        int lane, uint32_t tag) {
  const int K = P.K, NCd = P.NCd, NC = P.NC, b = pe.b;
  uint2* rec = P.dpart + static_cast<size_t>(b) * NCd;
  if (!stage_records(S.cbuf, rec, NCd, lane)) return false;
  __syncwarp();
  clear_records(rec, NCd, lane);
  for (int c = lane; c < NCd; c += 32) S.cmass[c] = ready_value(S.cbuf[c].y);
  __syncwarp();
  float W, rem;
  int chunk = pick_chunk(S.cmass, NCd, pe.u, lane, W, rem);
  __syncwarp();
  const float W_report = W;
  const uintptr_t rp = row_addr<DT>(P.target, static_cast<size_t>(b) * (K + 1) + pe.t_f, P.V);
  const uintptr_t rq = row_addr<DT>(P.draft, static_cast<size_t>(b) * K + pe.t_f, P.V);
  uint2* srec = P.part + (static_cast<size_t>(b) * P.R + pe.t_f) * NC;
  int tok = -1;
  Chunk kp, kq;
  if (W > 0.0f) {
    if (chunk >= 0 && ctl_fetch<DT>(P, S, cphase, rp, rq, chunk, kDrawBytes, true, kp, kq, lane))
      tok = draw_in_slot<DT>(reinterpret_cast<const unsigned char*>(S.cbuf), kp, kq, true, pe.prm,
                             rem, kDrawSweeps, lane);
  } else {
    // a residual of exactly zero mass: p's chunk masses from the stats records
    const float Mp = pe.prm.x, sT = pe.prm.z;
    for (int c = lane; c < NC; c += 32) {
      const uint2 r = ld_record(srec + c);
      const float m = __uint_as_float(r.x);
      S.cmass[c] = m > -INFINITY ? __fmul_rn(ready_value(r.y), scaled_exp(m, Mp, sT)) : 0.0f;
    }
    __syncwarp();
    float Wp;
    chunk = pick_chunk(S.cmass, NC, pe.u, lane, Wp, rem);
    const float4 prm = make_float4(Mp, 0.0f, sT, 0.0f);
    if (chunk >= 0 && ctl_fetch<DT>(P, S, cphase, rp, 0, chunk, kChunkBytes, false, kp, kq, lane))
      tok = draw_in_slot<DT>(reinterpret_cast<const unsigned char*>(S.cbuf), kp, kq, false, prm,
                             rem, kChunkBytes / 512, lane);
  }
  __syncwarp();
  clear_records(srec, NC, lane);
  if (P.row_stats && lane == 0) {
    float* rs = P.row_stats + (static_cast<size_t>(b) * (K + 1) + pe.t_f) * 8;
    rs[6] = __fdiv_rn(W_report, pe.Sp);
    rs[7] = static_cast<float>(tok);
  }
  if (tok < 0 || tok >= P.V) {
    finish_bad(P, b, SPECV_DEV_BAD_ROW, lane, tag);
  } else if (lane == 0) {
    P.out_tokens[static_cast<size_t>(b) * (K + 1) + pe.j] = tok;
  }
  __syncwarp();
  return true;
}

// ---------------------------------------------------------------- agent

// Asynchronous copies global -> shared: 16 bytes from L2 (never a stale L1
// line), 4 bytes of read-only input.  cp_async_arrive makes the barrier's
// current phase wait for every copy this thread issued before it, as one
// more arrival.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// The request window of a stats cursor: lane l describes request w0 + l.
struct Window {
  int w0;        // first request of the window
  int cnt;       // this lane's request: items
  int end;       // items up to and including this lane's request (INT_MAX past B)
  int n;         // draft length
  float sT;      // log2(e)/T, 0 for a greedy request
};

__device__ void load_window(const Params& P, Window& w, int w0, int base, int lane) {
  w.w0 = w0;
  const int b = w0 + lane;
  w.n = 0;
  w.sT = 0.0f;
  w.cnt = 0;
  if (b < P.B) {
    w.n = request_len(P, b);
    const float T = __ldg(P.temperature + b);
    w.cnt = request_items(P, w.n, T);
    if (w.cnt > 0 && T > 0.0f) w.sT = temp_scale(T);
  }
  const int incl = warp_incl_scan_int(w.cnt, lane);
  w.end = b < P.B ? base + incl : INT_MAX;
}

// Whole warp: maps stats item g to its request, row and chunk.  Returns
// false when g is past the last item.
__device__ bool map_item(const Params& P, Window& w, int g, int lane, Item& it) {
  for (;;) {
    const unsigned done = __ballot_sync(0xffffffffu, w.end <= g);
    if (done != 0xffffffffu) {
      const int i = __popc(done);   // ends are nondecreasing: `done` is a prefix
      if (w.w0 + i >= P.B) return false;
      const int end = __shfl_sync(0xffffffffu, w.end, i);
      const int cnt = __shfl_sync(0xffffffffu, w.cnt, i);
      const int n = __shfl_sync(0xffffffffu, w.n, i);
      const float sT = __shfl_sync(0xffffffffu, w.sT, i);
      const int local = g - (end - cnt);
      int r = __float2int_rz(__int2float_rn(local) * P.inv_NC);   // local < 2^24: exact operands
      if (r * P.NC > local) --r;
      if ((r + 1) * P.NC <= local) ++r;
      it.kind = kItemStats;
      it.b = w.w0 + i;
      it.c = local - r * P.NC;
      it.row = r <= n ? r : (P.K + 1) + (r - n - 1);
      it.mode = sT > 0.0f ? 0 : 1;
      it.sT = sT;
      const int t = r <= n ? r : r - n - 1;
      it.xrow = (sT > 0.0f && t < n) ? t : -1;
      return true;
    }
    const int last_end = __shfl_sync(0xffffffffu, w.end, 31);
    if (w.w0 + 32 >= P.B) return false;
    load_window(P, w, w.w0 + 32, last_end, lane);
  }
}

// Lane 0: stages an item into slot s of the agent's ring.  A draw item's
// decision fields come with it (cp.async on the slot's barrier).
template <int DT>
__device__ void issue(const Params& P, AgentSmem& A, unsigned char* slot, int s, const Item& it) {
  const int K = P.K;
  uintptr_t src0 = 0, src1 = 0;
  uint32_t n0 = 0, n1 = 0;
  unsigned char *dst0 = slot, *dst1 = slot;
  Item& dst = A.item[s];
  dst.kind = it.kind;
  dst.b = it.b;
  dst.row = it.row;
  dst.c = it.c;
  dst.mode = it.mode;
  dst.sT = it.sT;
  dst.xrow = it.xrow;
  dst.peek_b = it.peek_b;
  fence_proxy_async_smem();
  bool small = false;
  if (it.peek_b >= 0) {   // a sample of the draw cursor's request state
    cp_async16(&dst.peek, &P.req[it.peek_b].state);
    small = true;
  }
  if (it.kind == kItemStats && it.xrow >= 0) {
    cp_async4(&dst.x, P.draft_tokens + static_cast<size_t>(it.b) * K + it.xrow);
    small = true;
  }
  if (it.kind == kItemDraw) {
    cp_async16(&dst.prm, &P.req[it.b].prm);
    small = true;
  }
  if (small) cp_async_arrive(&A.full[s]);
  if (it.kind == kItemStats) {
    const bool is_draft = it.row > K;
    const uintptr_t row = is_draft
        ? row_addr<DT>(P.draft, static_cast<size_t>(it.b) * K + (it.row - K - 1), P.V)
        : row_addr<DT>(P.target, static_cast<size_t>(it.b) * (K + 1) + it.row, P.V);
    const Chunk k = chunk_of<DT>(row, P.V, it.c, kChunkBytes);
    n0 = bulk_span<DT>(k, is_draft ? P.d_lo : P.t_lo, is_draft ? P.d_hi : P.t_hi, &src0);
    if (n0) dst0 = slot + (src0 - k.g0);
  } else {
    const uintptr_t rp = row_addr<DT>(P.target, static_cast<size_t>(it.b) * (K + 1) + it.row, P.V);
    const Chunk kp = chunk_of<DT>(rp, P.V, it.c, kDrawBytes);
    n0 = bulk_span<DT>(kp, P.t_lo, P.t_hi, &src0);
    if (n0) dst0 = slot + (src0 - kp.g0);
    if (it.mode) {
      const uintptr_t rq = row_addr<DT>(P.draft, static_cast<size_t>(it.b) * K + it.row, P.V);
      const Chunk kq = draft_part<DT>(rq, kp);
      n1 = bulk_span<DT>(kq, P.d_lo, P.d_hi, &src1);
      if (n1) dst1 = slot + kDraftOff + (src1 - kq.g0);
    }
  }
  mbar_arrive_expect_tx(&A.full[s], n0 + n1);
  if (n0) bulk_copy_g2s(dst0, src0, n0, &A.full[s]);
  if (n1) bulk_copy_g2s(dst1, src1, n1, &A.full[s]);
}

// Whole warp: reduces the item in a slot and writes its record (lane 0).
template <int DT>
__device__ __forceinline__ void consume(const Params& P, unsigned char* slot, const Item& it,
                                        int lane) {
  const int K = P.K;
  if (it.kind == kItemStats) {
    const bool is_draft = it.row > K;
    const uintptr_t row = is_draft
        ? row_addr<DT>(P.draft, static_cast<size_t>(it.b) * K + (it.row - K - 1), P.V)
        : row_addr<DT>(P.target, static_cast<size_t>(it.b) * (K + 1) + it.row, P.V);
    const Chunk k = chunk_of<DT>(row, P.V, it.c, kChunkBytes);
    fix_edges<DT>(k, is_draft ? P.d_lo : P.t_lo, is_draft ? P.d_hi : P.t_hi, slot, lane);
    uint32_t lo, hi;
    if (it.mode) {
      const float2 r = chunk_argmax<DT>(slot, k, lane);
      lo = __float_as_uint(r.x);
      hi = __float_as_uint(r.y) | kReady;
    } else {
      const float2 r = chunk_softmax<DT>(slot, k, it.sT, lane);
      lo = __float_as_uint(r.x);
      hi = ready_bits(r.y);
    }
    if (lane == 0) {
      st_record(P.part + (static_cast<size_t>(it.b) * P.R + it.row) * P.NC + it.c, lo, hi);
      // the drafted token's logit, from the chunk that holds it
      if (it.xrow >= 0 && it.x >= k.e_lo && it.x < k.e_hi)
        st_record(P.zx + static_cast<size_t>(it.b) * P.R + it.row,
                  __float_as_uint(Elt<DT>::load(slot + k.off0 + it.x * Elt<DT>::kBytes)), kReady);
    }
  } else {
    const uintptr_t rp = row_addr<DT>(P.target, static_cast<size_t>(it.b) * (K + 1) + it.row, P.V);
    const Chunk kp = chunk_of<DT>(rp, P.V, it.c, kDrawBytes);
    fix_edges<DT>(kp, P.t_lo, P.t_hi, slot, lane);
    Chunk kq = kp;
    if (it.mode) {
      const uintptr_t rq = row_addr<DT>(P.draft, static_cast<size_t>(it.b) * K + it.row, P.V);
      kq = draft_part<DT>(rq, kp);
      fix_edges<DT>(kq, P.d_lo, P.d_hi, slot + kDraftOff, lane);
    }
    const float t = chunk_draw<DT>(slot, kp, kq, it.mode != 0, it.prm, lane);
    if (lane == 0) st_record(P.dpart + static_cast<size_t>(it.b) * P.NCd + it.c, 0u, ready_bits(t));
  }
}

template <int DT>
__device__ void agent(const Params& P, AgentSmem& A, unsigned char* ring, int lane, int aid,
                      int G, uint32_t tag) {
  Window w;
  load_window(P, w, 0, 0, lane);
  int g = aid;                       // next stats item
  bool stats_left = true;
  const int Dtot = P.B * P.NCd;      // < 2^31 within the size limits
  int d = aid;                       // next owned draw item
  int cur_b = d < Dtot ? d / P.NCd : -1;   // its request
  unsigned long long cur = 0;        // latest sample of that request's state
  int issued = 0, consumed = 0;
  bool ok = true;

  for (;;) {
    // ---- the draw cursor, from the latest state sample ------------------
    bool draw_ready = false;
    uint32_t payload = 0;
    if (d < Dtot && (cur >> 32) == tag) {
      const uint32_t pl = static_cast<uint32_t>(cur);
      if ((pl & 3u) == kStateDraws) {
        draw_ready = true;
        payload = pl;
        // the decision's fields were written before its state (release);
        // the draw items read them from L2 after this
        __threadfence();
      } else {
        // nothing to draw for this request: skip to an owned item past it
        const int nb = (cur_b + 1) * P.NCd;
        d += ((nb - d + G - 1) / G) * G;
        cur_b = d < Dtot ? d / P.NCd : -1;
        cur = 0;
      }
    }
    // ---- top up the ring without waiting -------------------------------
    while (issued - consumed < kSlots) {
      Item it;
      if (draw_ready) {
        it.kind = kItemDraw;
        it.b = cur_b;
        it.row = static_cast<int>((payload >> 3) & 31u);
        it.c = d - cur_b * P.NCd;
        it.mode = static_cast<int>((payload >> 2) & 1u);
        it.sT = 0.0f;
        it.xrow = -1;
        d += G;
        if (d >= Dtot || d / P.NCd != cur_b) {
          draw_ready = false;
          cur_b = d < Dtot ? d / P.NCd : -1;
          cur = 0;
        }
      } else if (stats_left) {
        if (!map_item(P, w, g, lane, it)) {
          stats_left = false;
          continue;
        }
        g += G;
      } else {
        break;
      }
      it.peek_b = (cur_b >= 0 && !draw_ready) ? cur_b : -1;   // sample it with this item
      const int s = issued % kSlots;
      __syncwarp();
      if (lane == 0) issue<DT>(P, A, ring + static_cast<size_t>(s) * kSlotBytes, s, it);
      ++issued;
    }

    if (issued == consumed) {
      // ring empty and no stats items left: poll the draw cursor's request
      if (d >= Dtot) break;
      const long long t0 = clock64();
      cur = ld_relaxed_u64(&P.req[cur_b].state);
      while ((cur >> 32) != tag) {
        __nanosleep(200);
        cur = ld_relaxed_u64(&P.req[cur_b].state);
        if (clock64() - t0 > kWaitLimitCycles) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      continue;
    }

    // ---- consume the oldest slot -----------------------------------------
    const int s = consumed % kSlots;
    const uint32_t ph = static_cast<uint32_t>(consumed / kSlots) & 1u;
    if (!warp_wait(&A.full[s], ph)) {
      ok = false;
      break;
    }
    const Item it = A.item[s];
    if (it.peek_b >= 0 && it.peek_b == cur_b && (it.peek >> 32) == tag) cur = it.peek;
    consume<DT>(P, ring + static_cast<size_t>(s) * kSlotBytes, it, lane);
    ++consumed;
  }
  if (!ok && lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
}

// ---------------------------------------------------------------- control

// The control warp of CTA x decides requests x, x + grid, x + 2 grid, ... in
// order, each once its stats records are all written, and draws the final
// token of each decided sampled request once its draw records are written
// (in decision order, up to kPend pending).  Requests whose length or
// temperature is unusable are answered first.
template <int DT>
__device__ void control(const Params& P, Smem& S, int lane, uint32_t tag) {
  const int x = static_cast<int>(blockIdx.x), grid = static_cast<int>(gridDim.x);
  // this CTA's requests' tokens and uniforms into L2 now, while the memory
  // system is idle; the decisions read them much later
  for (int b = x + lane * grid; b < P.B; b += 32 * grid) {
    prefetch_l2(P.draft_tokens + static_cast<size_t>(b) * P.K);
    prefetch_l2(P.uniforms + static_cast<size_t>(b) * (P.K + 1));
    prefetch_l2(P.uniforms_resample + b);
  }
  // unusable requests are answered now; greedy ones never have draw items,
  // which their owners learn from the state
  for (int base = x; base < P.B; base += 32 * grid) {
    const int b = base + lane * grid;
    int bad = 0;
    if (b < P.B) {
      const float T = __ldg(P.temperature + b);
      bad = request_bad(P, request_len(P, b), T);
      if (!bad && !(T > 0.0f)) set_state(P, b, tag, kStateNone);
    }
    for (unsigned m = __ballot_sync(0xffffffffu, bad != 0); m; m &= m - 1) {
      const int i = __ffs(m) - 1;
      finish_bad(P, base + i * grid, __shfl_sync(0xffffffffu, bad, i), lane, tag);
    }
  }
  uint32_t cphase = 0;   // phases of the control warp's chunk barrier
  int dec = x;              // next request to decide
  int dn = 0;               // its length and temperature
  float dT = 0.0f;
  bool dvalid = false;
  if (dec < P.B) {
    dn = request_len(P, dec);
    dT = __ldg(P.temperature + dec);
  }
  int ph = 0, pt = 0;       // pending draws [pt, ph)
  long long idle_since = clock64();
  bool ok = true;
  while (dec < P.B || pt < ph) {
    bool progress = false;
    if (dec < P.B && ph - pt < kPend) {
      dvalid = request_bad(P, dn, dT) == 0;
      int r = 1;
      if (dvalid) {
        Pend pe;
        r = try_decide<DT>(P, S, cphase, dec, dn, dT, lane, tag, pe);
        if (r == 2) {
          if (lane == 0) S.pend[ph % kPend] = pe;
          ++ph;
        }
      }
      if (r) {
        dec += grid;
        if (dec < P.B) {
          dn = request_len(P, dec);
          dT = __ldg(P.temperature + dec);
        }
        progress = true;
      }
      __syncwarp();
    }
    if (pt < ph) {
      const Pend pe = S.pend[pt % kPend];
      if (try_search<DT>(P, S, cphase, pe, lane, tag)) {
        ++pt;
        progress = true;
      }
      __syncwarp();
    }
    if (progress) {
      idle_since = clock64();
    } else {
      if (clock64() - idle_since > kWaitLimitCycles) {
        ok = false;
        break;
      }
      __nanosleep(128);
    }
  }
  if (!ok && lane == 0) atomicOr(P.header + kHStatus, SPECV_DEV_TIMEOUT);
}

// ---------------------------------------------------------------- kernel

template <int DT>
__global__ void __launch_bounds__(kThreads) verify_kernel(const Params P) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  __shared__ Smem S;
  extern __shared__ __align__(128) unsigned char dyn[];

  if (tid < kAgents * kSlots) mbar_init(&S.ag[tid / kSlots].full[tid % kSlots], 1);
  if (tid == 0) mbar_init(&S.cbar, 1);
  if (tid == 0) {
    S.tag = static_cast<uint32_t>(P.header[kHEpoch]) + 1u;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp < kAgents) {
    const int G = static_cast<int>(gridDim.x) * kAgents;
    const int aid = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
    agent<DT>(P, S.ag[warp], dyn + static_cast<size_t>(warp) * kSlots * kSlotBytes, tid & 31, aid,
              G, S.tag);
  } else {
    control<DT>(P, S, tid & 31, S.tag);
  }

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(P.header + kHExit, 1);
    if (prev == static_cast<int>(gridDim.x) - 1) {
      // last CTA of the launch: every item is done and every request
      // answered; reset for the next call
      P.header[kHExit] = 0;
      P.header[kHEpoch] = P.header[kHEpoch] + 1;
    }
  }
}

// ---------------------------------------------------------------- host side

int elt_bytes(specv_dtype dt) { return dt == SPECV_BF16 ? 2 : 4; }

struct Layout {
  size_t header, req, part, dpart, zx, total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Chunks per row for chunk size CB, for any 16-byte phase of the row.
int chunks_per_row(int V, specv_dtype dt, int CB) {
  return static_cast<int>((15 + static_cast<long long>(V) * elt_bytes(dt) + CB - 1) / CB);
}

Layout ws_layout(int B, int K, int V, specv_dtype dt) {
  const size_t R = 2 * static_cast<size_t>(K) + 1;
  const size_t NC = chunks_per_row(V, dt, kChunkBytes);
  const size_t NCd = chunks_per_row(V, dt, kDrawBytes);
  Layout L;
  L.header = 0;
  L.req = kHeaderBytes;
  L.part = align256(L.req + sizeof(Req) * static_cast<size_t>(B));
  L.dpart = align256(L.part + sizeof(uint2) * B * R * NC);
  L.zx = align256(L.dpart + sizeof(uint2) * static_cast<size_t>(B) * NCd);
  L.total = align256(L.zx + sizeof(uint2) * static_cast<size_t>(B) * R);
  return L;
}

// Resident CTAs of the kernel on the current device, cached per device.
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
    e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRingBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<DT>, kThreads,
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

// CTAs for a call: enough agents for the stats items of every row, at most
// the resident count.
int grid_for(int B, int K, int V, specv_dtype dtype, int ctas) {
  const long long items =
      static_cast<long long>(B) * (2 * K + 1) * chunks_per_row(V, dtype, kChunkBytes);
  long long want = (items + kAgents - 1) / kAgents;
  if (want < 1) want = 1;
  return static_cast<int>(want < ctas ? want : ctas);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uintptr_t up16(uintptr_t x) { return (x + 15) & ~static_cast<uintptr_t>(15); }
uintptr_t down16(uintptr_t x) { return x & ~static_cast<uintptr_t>(15); }

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

  int ctas = 0;
  if (resident_ctas_for(dtype, &ctas) != cudaSuccess || ctas < 1) return SPECV_ERR_CUDA;
  const int grid = grid_for(B, K, V, dtype, ctas);

  const Layout L = ws_layout(B, K, V, dtype);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  Params P;
  P.target = static_cast<const unsigned char*>(target);
  P.draft = static_cast<const unsigned char*>(draft);
  P.draft_tokens = draft_tokens;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.uniforms = uniforms;
  P.uniforms_resample = uniforms_resample;
  P.B = B;
  P.K = K;
  P.V = V;
  P.R = 2 * K + 1;
  P.NC = chunks_per_row(V, dtype, kChunkBytes);
  P.NCd = chunks_per_row(V, dtype, kDrawBytes);
  P.inv_NC = 1.0f / static_cast<float>(P.NC);
  const uintptr_t t0 = reinterpret_cast<uintptr_t>(target);
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(draft);
  P.t_lo = up16(t0);
  P.t_hi = down16(t0 + static_cast<size_t>(B) * (K + 1) * V * eb);
  P.d_lo = draft ? up16(d0) : 0;
  P.d_hi = draft ? down16(d0 + static_cast<size_t>(B) * K * V * eb) : 0;
  P.accepted_len = accepted_len;
  P.out_tokens = out_tokens;
  P.header = reinterpret_cast<int32_t*>(ws + L.header);
  P.req = reinterpret_cast<Req*>(ws + L.req);
  P.part = reinterpret_cast<uint2*>(ws + L.part);
  P.dpart = reinterpret_cast<uint2*>(ws + L.dpart);
  P.zx = reinterpret_cast<uint2*>(ws + L.zx);
  P.row_stats = row_stats;

  if (dtype == SPECV_BF16)
    verify_kernel<SPECV_BF16><<<grid, kThreads, kRingBytes, stream>>>(P);
  else
    verify_kernel<SPECV_F32><<<grid, kThreads, kRingBytes, stream>>>(P);
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

int specv_version(void) { return 400; }

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
