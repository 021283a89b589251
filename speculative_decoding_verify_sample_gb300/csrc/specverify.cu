// libspecverify: the speculative-decoding verification sampler for GB300
// (sm_103a).  One kernel does the whole step.
//
// The rule ("Decodificación Especulativa y EAGLE", Phase 10 - Lesson 25,
// sections "El Concepto", "La Regla de Exactitud", "Caso codicioso"): for
// each request, accept drafted tokens left to right while u_t < p(x_t)/q(x_t);
// at the first rejection draw a replacement from (p - q)+ and stop; if every
// draft is accepted draw a bonus token from p at the next position; at
// temperature 0 compare argmax(p) with the draft instead.
//
// Design.  Work unit = one (request b, position t).  A unit needs target row
// t, plus draft row t when t < n_b and T_b > 0.  Each unit is one
// thread-block cluster of C CTAs; CTA c owns vocabulary slice c and copies it
// from HBM into its shared memory once (TMA bulk copies, one mbarrier per
// row).  Everything else runs on chip:
//   1. slice maximum (raw logits) or slice argmax (greedy), combined across
//      the cluster through distributed shared memory;
//   2. slice sum of exp((z - max)/T), combined the same way -> p(x_t), q(x_t);
//   3. the accept test in log space;
//   4. if the unit's position could be the request's final draw (a rejected
//      position, or the bonus position), the inverse-CDF draw over the
//      residual (p - q)+ (or p) from the slices still in shared memory;
//   5. the unit's record {accept, candidate token} goes to the workspace and
//      the last unit of a request to arrive (atomic counter, no waiting)
//      scans the records and writes accepted_len and out_tokens.
// Every unit decides independently, so no unit waits for another; a unit
// whose candidate is not used costs only on-chip work.  Every logit the rule
// needs is read from HBM exactly once.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "specverify.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kSliceTargetBytes = 32 * 1024;   // per row per CTA
constexpr int kSliceMaxBytes = 96 * 1024;      // on-chip cap per row per CTA
constexpr int kChunkBytes = 16;                // one 128-bit vector
constexpr int kMaxTiles = kSliceMaxBytes / kChunkBytes / kThreads;   // 24
constexpr uint32_t kWaitLimit = 1u << 22;      // bounded mbarrier polling

constexpr int kRecAccept = 1;
constexpr int kRecBad = 2;

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
  int slice;               // elements per CTA slice (multiple of the chunk)
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t* status;
  int32_t* counters;       // [B]
  int2* records;           // [B, K+1]
  float* row_stats;        // [B, K+1, 8] or null
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
  __device__ static float load1(const void* base, size_t i) {
    return __ldg(static_cast<const float*>(base) + i);
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
  __device__ static float load1(const void* base, size_t i) {
    const unsigned short h = __ldg(static_cast<const unsigned short*>(base) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
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

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
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

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of the barrier, giving up after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 2^x on the MUFU unit (PTX ex2.approx.ftz.f32); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// ---------------------------------------------------------------- shared state

struct Xchg {             // slots other CTAs of the cluster read
  float max_p, max_q;     // phase 1
  int arg;                // phase 1 (greedy)
  int tmo;                // phase 1: this CTA's copy wait gave up
  float sum_p, sum_q;     // phase 2
  float w[2];             // phase 3 (and its p-fallback)
  int cand;               // phase 4: written by the owner CTA into rank 0
  int cand_set;
};

struct Smem {
  uint64_t bar[2];
  Xchg x;
  float red[2][kWarps];
  int redi[kWarps];
  float ws[kMaxTiles * kWarps];
  // request metadata, broadcast within the CTA
  int n, bad, tok, greedy, has_q, timeout, tmo_all;
  float T, u_t, u_bonus, u_res, zx_p, zx_q;
  // cluster-combined results
  float zmax_p, zmax_q, S_p, S_q;
  int gidx;
  int owner;
  float tau_owner;
  int sel_tile, sel_warp;
  float tau_warp;
  float W;
};

// ---------------------------------------------------------------- combine

// Called by thread 0 of cluster rank 0 after its unit's record is written.
// The last unit of request b to arrive scans the records and writes the
// outputs; no unit ever waits for another.
__device__ void arrive(const Params& P, int b, int n, bool timeout) {
  const int K = P.K;
  if (timeout) atomicOr(P.status, SPECV_DEV_TIMEOUT);
  __threadfence();
  const int prev = atomicAdd(P.counters + b, 1);
  if (prev != n) return;
  __threadfence();
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
    atomicOr(P.status, SPECV_DEV_BAD_ROW);
    P.accepted_len[b] = -1;
    for (int s = 0; s <= K; ++s) out[s] = -1;
  } else {
    const int final_tok = __ldcg(rec + j).x;
    for (int s = 0; s < j; ++s) out[s] = __ldg(P.draft_tokens + static_cast<size_t>(b) * K + s);
    out[j] = final_tok;
    for (int s = j + 1; s <= K; ++s) out[s] = -1;
    P.accepted_len[b] = j;
  }
  P.counters[b] = 0;   // leave the workspace ready for the next call
}

// ---------------------------------------------------------------- kernel

template <int DT>
struct Unit {
  using E = Elt<DT>;
  static constexpr int CH = E::kPerChunk;

  // Weight of element k of chunk c for the final draw: the residual
  // (p - q)+ scaled by S_p, or p scaled by S_p.
  __device__ static void chunk_weights(const unsigned char* bp, const unsigned char* bq, int c,
                                       int cnt, bool residual, float zmp, float zmq, float sT,
                                       float r, float w[CH]) {
    float vp[CH], vq[CH];
    E::unpack(reinterpret_cast<const uint4*>(bp)[c], vp);
    if (residual) E::unpack(reinterpret_cast<const uint4*>(bq)[c], vq);
    const int valid = cnt - c * CH;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const float ep = ex2(__fmul_rn(__fsub_rn(vp[k], zmp), sT));
      float wk = ep;
      if (residual) {
        const float eq = ex2(__fmul_rn(__fsub_rn(vq[k], zmq), sT));
        wk = fmaxf(__fmaf_rn(-r, eq, ep), 0.0f);
      }
      w[k] = k < valid ? wk : 0.0f;
    }
  }

  __device__ static float chunk_sum(const float w[CH]) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < CH; ++k) s = __fadd_rn(s, w[k]);
    return s;
  }
};

template <int DT>
__global__ void __launch_bounds__(kThreads) verify_kernel(const Params P) {
  using E = Elt<DT>;
  using U = Unit<DT>;
  constexpr int CH = E::kPerChunk;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int crank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int t = blockIdx.y;
  const int b = blockIdx.z;
  const int K = P.K, V = P.V;

  __shared__ Smem S;
  extern __shared__ __align__(128) unsigned char dyn[];
  const int slice_bytes_padded = ((P.slice * E::kBytes + 127) / 128) * 128;
  unsigned char* buf_p = dyn;
  unsigned char* buf_q = dyn + slice_bytes_padded;

  // ---- request metadata and validation (identical in every CTA) --------
  if (warp == 0) {
    const int n = P.draft_len ? __ldg(P.draft_len + b) : K;
    const float T = __ldg(P.temperature + b);
    int bad = 0;
    if (n < 1 || n > K) {
      bad |= SPECV_DEV_BAD_DRAFT_LEN;
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
    if (lane == 0) {
      S.n = n;
      S.bad = bad;
      S.T = T;
      S.timeout = 0;
      S.tmo_all = 0;
      S.x.cand = -1;
      S.x.cand_set = 0;
      if (!bad && t <= n) {
        S.greedy = (T == 0.0f);
        S.has_q = (T > 0.0f) && (t < n);
        S.tok = t < n ? __ldg(P.draft_tokens + static_cast<size_t>(b) * K + t) : -1;
        S.u_t = __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + t);
        S.u_bonus = __ldg(P.uniforms + static_cast<size_t>(b) * (K + 1) + n);
        S.u_res = __ldg(P.uniforms_resample + b);
      }
    }
  }
  __syncthreads();

  if (S.bad) {
    // Bad data: unit (b, 0) of cluster rank 0 writes the -1 outputs.
    if (t == 0 && crank == 0 && tid == 0) {
      atomicOr(P.status, S.bad);
      P.accepted_len[b] = -1;
      for (int s = 0; s <= K; ++s) P.out_tokens[static_cast<size_t>(b) * (K + 1) + s] = -1;
    }
    return;
  }
  const int n = S.n;
  if (t > n) return;      // rows after the draft are never read

  const bool greedy = S.greedy;
  const bool has_q = S.has_q;
  const size_t trow = (static_cast<size_t>(b) * (K + 1) + t) * static_cast<size_t>(V);
  const size_t drow = (static_cast<size_t>(b) * K + t) * static_cast<size_t>(V);
  const int e0 = crank * P.slice;
  const int cnt = max(0, min(P.slice, V - e0));
  const int nch = (cnt + CH - 1) / CH;

  // ---- stage the slice(s) into shared memory ---------------------------
  const unsigned char* gp = static_cast<const unsigned char*>(P.target) + (trow + e0) * E::kBytes;
  const unsigned char* gq =
      has_q ? static_cast<const unsigned char*>(P.draft) + (drow + e0) * E::kBytes : nullptr;
  const uint32_t bytes = static_cast<uint32_t>(cnt) * E::kBytes;
  const bool bulk_p = ((reinterpret_cast<uintptr_t>(gp) & 15) == 0) && ((bytes & 15) == 0);
  const bool bulk_q = has_q && ((reinterpret_cast<uintptr_t>(gq) & 15) == 0) && ((bytes & 15) == 0);

  if (tid == 0) {
    mbar_init(&S.bar[0], 1);
    mbar_init(&S.bar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) {
    if (bulk_p && bytes > 0) {
      mbar_expect_tx(&S.bar[0], bytes);
      bulk_copy_g2s(buf_p, gp, bytes, &S.bar[0]);
    }
    if (bulk_q && bytes > 0) {
      mbar_expect_tx(&S.bar[1], bytes);
      bulk_copy_g2s(buf_q, gq, bytes, &S.bar[1]);
    }
    // the drafted token's logits, for p(x_t) and q(x_t)
    if (!greedy && t < n) {
      S.zx_p = E::load1(P.target, trow + S.tok);
      S.zx_q = E::load1(P.draft, drow + S.tok);
    }
  }
  // Rows whose start is not 16-byte aligned: plain coalesced loads.
  if (!bulk_p) {
    for (int i = tid; i < cnt; i += kThreads) {
      if (DT == SPECV_F32)
        reinterpret_cast<float*>(buf_p)[i] = E::load1(P.target, trow + e0 + i);
      else
        reinterpret_cast<unsigned short*>(buf_p)[i] =
            __ldg(static_cast<const unsigned short*>(P.target) + trow + e0 + i);
    }
  }
  if (has_q && !bulk_q) {
    for (int i = tid; i < cnt; i += kThreads) {
      if (DT == SPECV_F32)
        reinterpret_cast<float*>(buf_q)[i] = E::load1(P.draft, drow + e0 + i);
      else
        reinterpret_cast<unsigned short*>(buf_q)[i] =
            __ldg(static_cast<const unsigned short*>(P.draft) + drow + e0 + i);
    }
  }
  bool ok = true;
  if (bulk_p && bytes > 0) ok &= mbar_wait_bounded(&S.bar[0], 0);
  if (bulk_q && bytes > 0) ok &= mbar_wait_bounded(&S.bar[1], 0);
  if (!ok) S.timeout = 1;   // benign race: every writer stores 1
  __syncthreads();

  // ---- phase 1: slice max / argmax --------------------------------------
  if (greedy) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int c = tid; c < nch; c += kThreads) {
      float v[CH];
      E::unpack(reinterpret_cast<const uint4*>(buf_p)[c], v);
      const int valid = cnt - c * CH;
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int idx = e0 + c * CH + k;
        if (k < valid && better(v[k], idx, bv, bi)) { bv = v[k]; bi = idx; }
      }
    }
    warp_argmax(bv, bi);
    if (lane == 0) { S.red[0][warp] = bv; S.redi[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
      bv = lane < kWarps ? S.red[0][lane] : -INFINITY;
      bi = lane < kWarps ? S.redi[lane] : INT_MAX;
      warp_argmax(bv, bi);
      if (lane == 0) { S.x.max_p = bv; S.x.arg = bi; S.x.tmo = S.timeout; }
    }
    cluster.sync();
    if (warp == 0) {
      float v = -INFINITY;
      int i = INT_MAX, tmo = 0;
      if (lane < C) {
        const Xchg* rx = cluster.map_shared_rank(&S.x, lane);
        v = rx->max_p;
        i = rx->arg;
        tmo = rx->tmo;
      }
      warp_argmax(v, i);
      tmo = __any_sync(0xffffffffu, tmo);
      if (lane == 0) { S.zmax_p = v; S.gidx = i; S.tmo_all = tmo; }
    }
    cluster.sync();   // remote reads done before any CTA exits
    if (crank == 0 && tid == 0) {
      const int g = S.gidx;
      int flags = (t < n && g == S.tok) ? kRecAccept : 0;
      if (g < 0 || g >= V || S.tmo_all) flags |= kRecBad;
      if (P.row_stats) {
        float* rs = P.row_stats + (static_cast<size_t>(b) * (K + 1) + t) * 8;
        rs[0] = S.zmax_p;
        rs[7] = static_cast<float>(g);
      }
      P.records[static_cast<size_t>(b) * (K + 1) + t] = make_int2(g, flags);
      arrive(P, b, n, S.tmo_all);
    }
    return;
  }

  {
    float mp = -INFINITY, mq = -INFINITY;
    for (int c = tid; c < nch; c += kThreads) {
      float v[CH];
      const int valid = cnt - c * CH;
      E::unpack(reinterpret_cast<const uint4*>(buf_p)[c], v);
#pragma unroll
      for (int k = 0; k < CH; ++k)
        if (k < valid) mp = fmaxf(mp, v[k]);
      if (has_q) {
        E::unpack(reinterpret_cast<const uint4*>(buf_q)[c], v);
#pragma unroll
        for (int k = 0; k < CH; ++k)
          if (k < valid) mq = fmaxf(mq, v[k]);
      }
    }
    mp = warp_max(mp);
    mq = warp_max(mq);
    if (lane == 0) { S.red[0][warp] = mp; S.red[1][warp] = mq; }
    __syncthreads();
    if (warp == 0) {
      mp = warp_max(lane < kWarps ? S.red[0][lane] : -INFINITY);
      mq = warp_max(lane < kWarps ? S.red[1][lane] : -INFINITY);
      if (lane == 0) { S.x.max_p = mp; S.x.max_q = mq; S.x.tmo = S.timeout; }
    }
    cluster.sync();
    if (warp == 0) {
      float a = -INFINITY, c2 = -INFINITY;
      int tmo = 0;
      if (lane < C) {
        const Xchg* rx = cluster.map_shared_rank(&S.x, lane);
        a = rx->max_p;
        c2 = rx->max_q;
        tmo = rx->tmo;
      }
      a = warp_max(a);
      c2 = warp_max(c2);
      tmo = __any_sync(0xffffffffu, tmo);
      if (lane == 0) { S.zmax_p = a; S.zmax_q = c2; S.tmo_all = tmo; }
    }
    __syncthreads();

    // ---- phase 2: sums of exp((z - max)/T) -------------------------------
    const float sT = __fdiv_rn(kLog2e, S.T);
    const float zmp = S.zmax_p, zmq = S.zmax_q;
    float sp = 0.0f, sq = 0.0f;
    for (int c = tid; c < nch; c += kThreads) {
      float v[CH];
      const int valid = cnt - c * CH;
      E::unpack(reinterpret_cast<const uint4*>(buf_p)[c], v);
#pragma unroll
      for (int k = 0; k < CH; ++k)
        if (k < valid) sp = __fadd_rn(sp, ex2(__fmul_rn(__fsub_rn(v[k], zmp), sT)));
      if (has_q) {
        E::unpack(reinterpret_cast<const uint4*>(buf_q)[c], v);
#pragma unroll
        for (int k = 0; k < CH; ++k)
          if (k < valid) sq = __fadd_rn(sq, ex2(__fmul_rn(__fsub_rn(v[k], zmq), sT)));
      }
    }
    sp = warp_sum(sp);
    sq = warp_sum(sq);
    if (lane == 0) { S.red[0][warp] = sp; S.red[1][warp] = sq; }
    __syncthreads();
    if (warp == 0) {
      sp = warp_sum(lane < kWarps ? S.red[0][lane] : 0.0f);
      sq = warp_sum(lane < kWarps ? S.red[1][lane] : 0.0f);
      if (lane == 0) { S.x.sum_p = sp; S.x.sum_q = sq; }
    }
    cluster.sync();
    if (warp == 0) {
      float a = 0.0f, c2 = 0.0f;
      if (lane < C) {
        const Xchg* rx = cluster.map_shared_rank(&S.x, lane);
        a = rx->sum_p;
        c2 = rx->sum_q;
      }
      a = warp_sum(a);
      c2 = warp_sum(c2);
      if (lane == 0) { S.S_p = a; S.S_q = c2; }
    }
    __syncthreads();

    // ---- phase 3: the accept test (log2 domain) ---------------------------
    const float Sp = S.S_p, Sq = S.S_q;
    // identical in every CTA of the cluster: it steers cluster barriers
    const bool row_ok = isfinite(zmp) && (!has_q || isfinite(zmq)) && !S.tmo_all;
    bool accept = false;
    float lp = 0.0f, lq = 0.0f;
    if (t < n) {
      lp = __fsub_rn(__fmul_rn(__fsub_rn(S.zx_p, zmp), sT), log2f(Sp));
      lq = __fsub_rn(__fmul_rn(__fsub_rn(S.zx_q, zmq), sT), log2f(Sq));
      accept = __fadd_rn(log2f(S.u_t), lq) < lp;
    }
    const bool want_draw = row_ok && ((t == n) || !accept || P.row_stats != nullptr);
    int cand = -1;
    float Wtot = 0.0f;

    if (want_draw) {
      // ---- phase 4: inverse-CDF draw over the on-chip slices ----------------
      bool residual = (t < n);
      float u = residual ? S.u_res : S.u_bonus;
      const float r = __fdiv_rn(Sp, Sq);
      const int ntiles = (nch + kThreads - 1) / kThreads;
      int owner = -1;
      for (int attempt = 0; attempt < 2; ++attempt) {
        // per tile, per warp partial sums in index order
        for (int tile = 0; tile < ntiles; ++tile) {
          const int c = tile * kThreads + tid;
          float w[CH];
          float s = 0.0f;
          if (c < nch) {
            U::chunk_weights(buf_p, buf_q, c, cnt, residual, zmp, zmq, sT, r, w);
            s = U::chunk_sum(w);
          }
          const float incl = warp_incl_scan(s, lane);
          if (lane == 31) S.ws[tile * kWarps + warp] = incl;
        }
        __syncthreads();
        if (tid == 0) {
          float Wc = 0.0f;
          for (int k = 0; k < ntiles * kWarps; ++k) Wc = __fadd_rn(Wc, S.ws[k]);
          S.x.w[attempt] = Wc;
        }
        cluster.sync();
        if (warp == 0) {
          float wc = 0.0f;
          if (lane < C) wc = cluster.map_shared_rank(&S.x, lane)->w[attempt];
          const float incl = warp_incl_scan(wc, lane);
          const float W = __shfl_sync(0xffffffffu, incl, 31);
          const float tau = __fmul_rn(u, W);
          const unsigned hit = __ballot_sync(0xffffffffu, lane < C && wc > 0.0f && incl > tau);
          const unsigned pos = __ballot_sync(0xffffffffu, lane < C && wc > 0.0f);
          const int own = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
          const float excl = __shfl_sync(0xffffffffu, incl, own > 0 ? own - 1 : 0);
          if (lane == 0) {
            S.W = W;
            S.owner = own;
            S.tau_owner = __fsub_rn(tau, own > 0 ? excl : 0.0f);
          }
        }
        __syncthreads();
        owner = S.owner;
        const float W_attempt = S.W;
        if (attempt == 0) Wtot = W_attempt;   // reported mass: before any fallback
        if (!(residual && !(W_attempt > 0.0f))) break;
        // residual of exactly zero mass: draw from p with the same uniform
        residual = false;
      }

      if (owner == crank) {
        if (tid == 0) {
          const float tau1 = S.tau_owner;
          float acc = 0.0f, sel_acc = 0.0f, last_acc = 0.0f;
          int sel = -1, last = -1;
          for (int k = 0; k < ntiles * kWarps; ++k) {
            const float wk = S.ws[k];
            if (wk > 0.0f) {
              if (__fadd_rn(acc, wk) > tau1) { sel = k; sel_acc = acc; break; }
              last = k;
              last_acc = acc;
            }
            acc = __fadd_rn(acc, wk);
          }
          if (sel < 0) { sel = last; sel_acc = last_acc; }
          S.sel_tile = sel / kWarps;
          S.sel_warp = sel % kWarps;
          S.tau_warp = __fsub_rn(tau1, sel_acc);
        }
        __syncthreads();
        if (warp == S.sel_warp) {
          const int c = S.sel_tile * kThreads + tid;
          float w[CH];
          float s = 0.0f;
          if (c < nch) {
            U::chunk_weights(buf_p, buf_q, c, cnt, residual, zmp, zmq, sT, r, w);
            s = U::chunk_sum(w);
          } else {
#pragma unroll
            for (int k = 0; k < CH; ++k) w[k] = 0.0f;
          }
          const float incl = warp_incl_scan(s, lane);
          const float tau2 = S.tau_warp;
          const unsigned hit = __ballot_sync(0xffffffffu, s > 0.0f && incl > tau2);
          const unsigned pos = __ballot_sync(0xffffffffu, s > 0.0f);
          const int l = hit ? __ffs(hit) - 1 : 31 - __clz(pos);
          const float excl = __shfl_up_sync(0xffffffffu, incl, 1);
          if (lane == l) {
            const float tau3 = __fsub_rn(tau2, l > 0 ? excl : 0.0f);
            float run = 0.0f;
            int pick = -1, lastk = -1;
#pragma unroll
            for (int k = 0; k < CH; ++k) {
              if (w[k] > 0.0f) {
                run = __fadd_rn(run, w[k]);
                if (pick < 0 && run > tau3) pick = k;
                lastk = k;
              }
            }
            if (pick < 0) pick = lastk;
            Xchg* r0 = cluster.map_shared_rank(&S.x, 0);
            r0->cand = e0 + c * CH + pick;
            r0->cand_set = 1;
          }
        }
      }
      cluster.sync();   // candidate visible in rank 0; remote accesses done
      cand = (crank == 0) ? S.x.cand : -1;
    } else {
      cluster.sync();   // remote reads done before any CTA exits
    }

    if (crank == 0 && tid == 0) {
      int flags = accept ? kRecAccept : 0;
      if (!row_ok) flags |= kRecBad;
      if (want_draw && (cand < 0 || cand >= V)) flags |= kRecBad;
      if (P.row_stats) {
        float* rs = P.row_stats + (static_cast<size_t>(b) * (K + 1) + t) * 8;
        rs[0] = zmp;
        rs[1] = Sp;
        if (t < n) {
          rs[2] = lp * kLn2;
          rs[3] = zmq;
          rs[4] = Sq;
          rs[5] = lq * kLn2;
        }
        rs[6] = __fdiv_rn(Wtot, Sp);
        rs[7] = static_cast<float>(cand);
      }
      P.records[static_cast<size_t>(b) * (K + 1) + t] = make_int2(cand, flags);
      arrive(P, b, n, S.tmo_all);
    }
  }

}

// ---------------------------------------------------------------- host side

struct Plan {
  int C;       // cluster size (CTAs per unit)
  int slice;   // elements per CTA
  size_t smem; // dynamic shared memory bytes
};

int elt_bytes(specv_dtype dt) { return dt == SPECV_BF16 ? 2 : 4; }

bool make_plan(int V, specv_dtype dt, bool with_draft, Plan* plan) {
  const int eb = elt_bytes(dt);
  const int per_chunk = kChunkBytes / eb;
  const long long row_bytes = static_cast<long long>(V) * eb;
  long long C = (row_bytes + kSliceTargetBytes - 1) / kSliceTargetBytes;
  if (C < 1) C = 1;
  if (C > kMaxCluster) C = kMaxCluster;
  long long slice = (V + C - 1) / C;
  slice = (slice + per_chunk - 1) / per_chunk * per_chunk;
  if (slice * eb > kSliceMaxBytes) return false;
  C = (V + slice - 1) / slice;
  const size_t padded = static_cast<size_t>((slice * eb + 127) / 128 * 128);
  plan->C = static_cast<int>(C);
  plan->slice = static_cast<int>(slice);
  plan->smem = with_draft ? 2 * padded : padded;
  return true;
}

template <int DT>
cudaError_t configure_kernel() {
  // Per-process, per-device attribute setup; idempotent.
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           2 * kSliceMaxBytes + 256);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) done[dev] = true;
  return cudaSuccess;
}

size_t ws_status_bytes() { return 16; }
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
  P.slice = plan.slice;
  P.accepted_len = accepted_len;
  P.out_tokens = out_tokens;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  P.status = reinterpret_cast<int32_t*>(ws);
  P.counters = reinterpret_cast<int32_t*>(ws + ws_status_bytes());
  P.records = reinterpret_cast<int2*>(ws + ws_status_bytes() + ws_counter_bytes(B));
  P.row_stats = row_stats;

  cudaError_t e = dtype == SPECV_BF16 ? configure_kernel<SPECV_BF16>() : configure_kernel<SPECV_F32>();
  if (e != cudaSuccess) return SPECV_ERR_CUDA;

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(plan.C), static_cast<unsigned>(K + 1),
                     static_cast<unsigned>(B));
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
// workspace (status word, per-request counters, per-unit records), sized for
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
  return ws_status_bytes() + ws_counter_bytes(B) + static_cast<size_t>(B) * (K + 1) * 8;
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
  if (!workspace || !status || workspace_bytes < ws_status_bytes()) return SPECV_ERR_INVALID_ARG;
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
