// flce_gemm.cuh — the persistent, warp-specialised tcgen05 GEMM that every
// product of the fused linear cross-entropy runs on, and its epilogues.
//
//   warp 8      TMA producer: fills a shared-memory ring with 128-byte swizzled
//               bf16 tiles of A and B (4 stages of 128x64 + 256x64 for one CTA;
//               6 stages of 128x64 + its 128x64 half of B per CTA of a pair).
//   warp 9      MMA issuer: one elected thread issues tcgen05.mma (M=128 or,
//               for a CTA pair, M=256; N=256; K=16) into one of two TMEM
//               accumulators (2 x 256 fp32 columns) and commits stage releases
//               and accumulator-ready signals to mbarriers.  The whole warp owns
//               the TMEM allocation.
//   warps 0-7   two epilogue groups in ping-pong: group g owns accumulator g
//               and takes every other tile; thread i of a group owns TMEM lane i
//               (one output row) and reads 32 columns at a time with tcgen05.ld.
//
// Epilogue policies:
//   EpiFwd    logits -> bias, scale, soft cap -> online (max, sum exp,
//             sum exp*z, argmax, target logit) per token across a vocabulary
//             split, one record per (split, group, token); optionally keeps z.
//   EpiGrad   recomputed logits -> G = w_n (softmax - onehot) dz/dacc in bf16
//             for one vocabulary chunk, plus per-tile dbias column sums.
//   EpiStore  accumulator -> bf16 / fp32 store (dW; the test GEMM).
//   EpiAccum  accumulator -> fp32 slot (=, +=) or the final store (dh; dW of
//             the token-chunked backward).
//
// Every wait is bounded (see mbar_wait); a role that gives up raises a
// CTA-wide abort flag, the others stop at their next wait, in-flight copies
// and MMAs are drained, TMEM is freed and the kernel returns with
// FLCE_ERR_TIMEOUT in the device status word.
#pragma once

#include <cuda.h>
#include <cfloat>

#include "flce_device.cuh"
#include "flce_internal.h"

namespace flce {

struct Unit {
  int m_blk, n_unit, n_first, n_count, kb_first, kb_count, ks;
  int64_t row0;  // first output row of this CTA's 128-row slice of the tile
  bool skip;     // the tile starts past the device-side row limit: no work
};

// Device-side limits of a launch (valid-token compaction), read once.  With a
// row limit the units are enumerated over the m tiles that hold a valid row
// only, so the persistent CTAs stay balanced.
struct Limits {
  int32_t m_rows;       // rows at or past this hold no work
  int32_t m_tiles;      // m tiles enumerated
  int32_t total_units;  // units enumerated
  int32_t k_blocks;     // K blocks past this are not loaded or multiplied
};
__device__ __forceinline__ Limits read_limits(const GemmSched& sc, int rows_per_tile) {
  Limits l;
  l.m_rows = 0x7fffffff;
  l.m_tiles = sc.m_tiles;
  l.total_units = sc.total_units;
  if (sc.m_limit) {
    l.m_rows = *reinterpret_cast<const volatile int32_t*>(sc.m_limit);
    l.m_tiles = min(sc.m_tiles, (l.m_rows + rows_per_tile - 1) / rows_per_tile);
    l.total_units = l.m_tiles * sc.n_units * sc.ksplit;
  }
  l.k_blocks = sc.k_limit ? (*reinterpret_cast<const volatile int32_t*>(sc.k_limit) + kBK - 1) / kBK : 0x7fffffff;
  return l;
}

__device__ __forceinline__ Unit decode_unit(const GemmSched& sc, int u, int rows_per_tile, uint32_t rank,
                                            const Limits& lim) {
  const int per_m = sc.n_units * sc.ksplit;
  const int per_group = sc.group_m * per_m;
  const int g = u / per_group;
  const int r = u - g * per_group;
  const int m0 = g * sc.group_m;
  const int gm = min(sc.group_m, lim.m_tiles - m0);
  const int m_local = r % gm;
  const int rest = r / gm;
  Unit t;
  t.m_blk = m0 + m_local;
  if (sc.ks_outer) {  // units running together share one K slice (long K, operands far beyond L2)
    t.n_unit = rest % sc.n_units;
    t.ks = rest / sc.n_units;
  } else {
    t.ks = rest % sc.ksplit;
    t.n_unit = rest / sc.ksplit;
  }
  t.n_first = t.n_unit * sc.n_per_unit;
  t.n_count = min(sc.n_per_unit, sc.n_tiles - t.n_first);
  t.kb_first = t.ks * sc.kb_per_split;
  t.kb_count = max(0, min(sc.kb_per_split, min(sc.k_blocks, lim.k_blocks) - t.kb_first));
  t.row0 = static_cast<int64_t>(t.m_blk) * rows_per_tile + static_cast<int64_t>(rank) * kBM;
  t.skip = static_cast<int64_t>(t.m_blk) * rows_per_tile >= lim.m_rows;
  return t;
}

__device__ __forceinline__ float load_bias(const void* bias, int bias_f32, int64_t v) {
  if (bias_f32) return __ldg(reinterpret_cast<const float*>(bias) + v);
  const unsigned short raw = __ldg(reinterpret_cast<const unsigned short*>(bias) + v);
  return __uint_as_float(static_cast<uint32_t>(raw) << 16);
}

// The 32 bias values of columns [vc, vc+32) (0 past the vocabulary).  Every
// lane reads the same addresses, so each load is one broadcast transaction;
// 16-byte vectors when the bias is aligned and the chunk is whole.
__device__ __forceinline__ void load_bias_chunk(const void* bias, int bias_f32, int bias_vec, int64_t vc,
                                                int64_t vocab, float (&b)[32]) {
  if (bias_vec && vc + 32 <= vocab) {
    if (bias_f32) {
      const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(bias) + vc);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = __ldg(src + q);
        b[4 * q] = v.x;
        b[4 * q + 1] = v.y;
        b[4 * q + 2] = v.z;
        b[4 * q + 3] = v.w;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(bias) + vc);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldg(src + q);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          b[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
          b[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) b[j] = (vc + j < vocab) ? load_bias(bias, bias_f32, vc + j) : 0.f;
  }
}

// Runs f(r, c) over the first `nch` 32-column chunks of this warp's TMEM
// lanes.  kPipelined: chunk c+1 is loaded while chunk c is processed (for the
// light epilogues; the heavy ones leave the registers to the math and rely on
// the other epilogue group for overlap).  nch is warp-uniform.
template <bool kPipelined = true, class F>
__device__ __forceinline__ void for_each_tmem_chunk(uint32_t taddr, int nch, F&& f) {
  if (nch <= 0) return;
  if (!kPipelined) {
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait(r);
      f(r, c);
    }
    return;
  }
  uint32_t ra[32], rb[32];
  tmem_ld32(taddr, ra);
  tmem_ld_wait(ra);
#pragma unroll 1
  for (int c = 0; c < nch; c += 2) {
    const bool has1 = c + 1 < nch;
    if (has1) tmem_ld32(taddr + (c + 1) * 32, rb);
    f(ra, c);
    if (has1) {
      tmem_ld_wait(rb);
      const bool has2 = c + 2 < nch;
      if (has2) tmem_ld32(taddr + (c + 2) * 32, ra);
      f(rb, c + 1);
      if (has2) tmem_ld_wait(ra);
    }
  }
}

// Number of 32-column chunks of a tile that start inside [0, limit).
__device__ __forceinline__ int chunks_below(int64_t col0, int64_t limit) {
  const int64_t rem = limit - col0;
  if (rem <= 0) return 0;
  return rem >= kBN ? kBN / 32 : static_cast<int>((rem + 31) / 32);
}

// The 128 threads of one epilogue group agree on a predicate (named barrier
// `id`, AND).
__device__ __forceinline__ bool epilogue_all(bool ok, int id) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok)), "r"(id), "n"(kEpilogueThreads)
      : "memory");
  return r != 0;
}

// Thread index within its epilogue group (its TMEM lane, i.e. its tile row).
__device__ __forceinline__ int epi_tid() { return static_cast<int>(threadIdx.x) & (kEpilogueThreads - 1); }

__device__ __forceinline__ float max32(const float (&z)[32]) {  // 16 three-input maxima
  float t[10];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = max3f(z[3 * i], z[3 * i + 1], z[3 * i + 2]);
  const float u = max3f(z[30], z[31], t[0]);
  const float a = max3f(t[1], t[2], t[3]), b = max3f(t[4], t[5], t[6]), c = max3f(t[7], t[8], t[9]);
  return fmaxf(max3f(a, b, c), u);
}

// ============================================================================
// Epilogue: forward statistics over one vocabulary split
// ============================================================================
// Stages this warp's box of 32 rows x 128 bytes (lane = row; r = the row's 32
// words: 32 fp32 values, or 64 bf16 values packed in pairs) in `buf` with the
// tensor map's 128-byte swizzle (16-byte chunk j of row r lands at chunk
// j ^ (r mod 8)), then lane 0 stores it with TMA at (col, row_base); the map
// clips rows and columns outside the tensor.  buf: kStoreStageBytes,
// 1024-byte aligned.
__device__ __forceinline__ void store_box_tma(const CUtensorMap* map, uint8_t* buf, int64_t col, int64_t row_base,
                                              const uint32_t (&r)[32]) {
  const uint32_t lane = lane_id();
  if (lane == 0) bulk_wait_read_all();  // the previous box has left this buffer
  __syncwarp();
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(row + ((j ^ (lane & 7)) * 16), r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, static_cast<int32_t>(col), static_cast<int32_t>(row_base));
    bulk_commit_group();
  }
}

// This warp's staging buffer (one per epilogue warp, in the epilogue region
// whose group slice is epi_smem).
__device__ __forceinline__ uint8_t* warp_stage_buffer(float* epi_smem, int grp) {
  return reinterpret_cast<uint8_t*>(epi_smem - grp * kEpiSmemGroupFloats) + (threadIdx.x >> 5) * kStoreStageBytes;
}

// Every box this warp stored is complete.
__device__ __forceinline__ void finish_box_stores() {
  if (lane_id() == 0) bulk_wait_all();
  __syncwarp();
}

template <bool kBias, bool kSoftcap>
struct EpiFwd {
  using Params = FwdParams;
  // Staging of the kept logits (TMA stores), one buffer per epilogue warp.
  static constexpr int kTailBytes = kEpilogueGroups * kEpilogueWarps * kStoreStageBytes;
  __device__ static void finish(const Params& p) {
    if (p.z_out) finish_box_stores();
  }
  struct State {
    int64_t row, target;
    float m, s, a, best, zt;
    int32_t best_idx;
    bool has_zt;  // this group processed the tile holding the target
  };

  __device__ static void begin_unit(const Params& p, const Unit& u, State& st, int /*grp*/) {
    st.row = u.row0 + epi_tid();
    st.target = st.row < p.n_tokens ? __ldg(p.targets + st.row) : p.ignore_index;
    st.m = -INFINITY;
    st.s = 0.f;
    st.a = 0.f;
    st.best = -INFINITY;
    st.best_idx = 0;
    st.zt = 0.f;
    st.has_zt = false;
  }

  __device__ static void tile(const Params& p, const Unit& u, int n_tile, uint32_t taddr, State& st,
                              float* epi_smem, int grp) {
    const int64_t v_tile = static_cast<int64_t>(n_tile) * kBN;
    // Kept logits: this warp's 32 rows go out as 32 x 32 boxes (the map clips rows past the chunk).
    const int64_t row_base = u.row0 + ((threadIdx.x >> 5) % kEpilogueWarps) * 32;
    const bool keep_z = p.z_out != nullptr && row_base < p.n_tokens;
    uint8_t* zbuf = warp_stage_buffer(epi_smem, grp);
    // z = c tanh(s x / c) = c - 2c / (2^t + 1) with t = 2 (s x / c) log2 e = x k_t.  The
    // arithmetic runs on packed fp32 pairs (columns j, j + 1).
    const uint64_t k_t2 = f2_splat(p.scale * p.inv_softcap * 2.0f * kLog2e);
    const uint64_t scale2 = f2_splat(p.scale);
    const uint64_t cap2 = f2_splat(p.softcap), m2cap2 = f2_splat(-2.0f * p.softcap);
    for_each_tmem_chunk<false>(taddr, chunks_below(v_tile, p.vocab), [&](const uint32_t (&r)[32], int c) {
      const int64_t vc = v_tile + c * 32;
      const bool ragged = vc + 32 > p.vocab;
      float bch[32];
      if (kBias) load_bias_chunk(p.bias, p.bias_f32, p.bias_vec, vc, p.vocab, bch);
      float z[32];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        uint64_t x = f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
        if (kBias) x = f2_add(x, f2_pack(bch[j], bch[j + 1]));
        if (kSoftcap) {  // the reciprocal pair comes back swapped: low lane = column j + 1
          float t0, t1;
          f2_unpack(f2_mul(x, k_t2), t0, t1);
          f2_unpack(f2_fma(f2_inv_exp2p1_swapped(t0, t1), m2cap2, cap2), z[j + 1], z[j]);
        } else {
          f2_unpack(f2_mul(x, scale2), z[j], z[j + 1]);
        }
      }
      if (keep_z) {  // keep the logits for the token-chunked backward
        uint32_t zb[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) zb[j] = __float_as_uint(z[j]);
        store_box_tma(&p.z_map, zbuf, vc, row_base, zb);
      }
      if (ragged) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (vc + j >= p.vocab) z[j] = -FLT_MAX;
      }
      const float cmax = max32(z);
      if (cmax > st.best) {  // strict: the lowest index wins ties, across chunks and tiles
        int jj = 31;
#pragma unroll
        for (int j = 31; j >= 0; --j)
          if (z[j] == cmax) jj = j;
        st.best = cmax;
        st.best_idx = static_cast<int32_t>(vc + jj);
      }
      if (cmax > st.m) {  // lazy rescale of the running sums to the new maximum
        const float f = ex2_approx((st.m - cmax) * kLog2e);
        st.s *= f;
        st.a *= f;
        st.m = cmax;
      }
      // Four partial sums per chunk (columns j mod 4), two packed pairs each.  The pairs keep the
      // lane order the z arithmetic left them in (low lane = column j + kLo).
      constexpr int kLo = kSoftcap ? 1 : 0;
      const uint64_t l2e2 = f2_splat(kLog2e), nmb2 = f2_splat(-st.m * kLog2e);
      uint64_t s2[2] = {0ull, 0ull}, a2[2] = {0ull, 0ull};
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const uint64_t zz = f2_pack(z[j + kLo], z[j + 1 - kLo]);
        float u0, u1;
        f2_unpack(f2_fma(zz, l2e2, nmb2), u0, u1);
        const uint64_t e = f2_pack(ex2_approx(u0), ex2_approx(u1));
        s2[(j >> 1) & 1] = f2_add(s2[(j >> 1) & 1], e);
        a2[(j >> 1) & 1] = f2_fma(e, zz, a2[(j >> 1) & 1]);
      }
      float s4[4], a4[4];
      f2_unpack(s2[0], s4[kLo], s4[1 - kLo]);
      f2_unpack(s2[1], s4[2 + kLo], s4[3 - kLo]);
      f2_unpack(a2[0], a4[kLo], a4[1 - kLo]);
      f2_unpack(a2[1], a4[2 + kLo], a4[3 - kLo]);
      st.s += (s4[0] + s4[1]) + (s4[2] + s4[3]);
      st.a += (a4[0] + a4[1]) + (a4[2] + a4[3]);
      const int64_t tl = st.target - vc;
      if (tl >= 0 && tl < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == tl) st.zt = z[j];
        st.has_zt = true;
      }
    });
  }

  __device__ static void end_unit(const Params& p, const Unit& u, State& st, int grp) {
    if (st.row >= p.n_tokens) return;
    const size_t rec = static_cast<size_t>(u.n_unit) * kEpilogueGroups + grp;
    const size_t o = rec * static_cast<size_t>(p.n_tokens) + st.row;
    p.part_m[o] = st.m;
    p.part_s[o] = st.s;
    p.part_a[o] = st.a;
    p.part_best[o] = st.best;
    p.part_idx[o] = st.best_idx;
    if (st.has_zt) p.z_target[st.row] = st.zt;
  }
};

// ============================================================================
// Epilogue: backward logit gradient G for one vocabulary chunk
// ============================================================================
// Reduce 32 per-lane column values over the 32 lanes of the warp; afterwards
// lane l holds the sum of column l over the warp's 32 rows (fixed order).
__device__ __forceinline__ float warp_column_sums(float (&v)[32]) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// Upstream weight w_n of a valid token: dloss[n] (none), dloss (sum) or
// dloss / denominator (mean; num_items when > 0, else the valid count).
__device__ __forceinline__ float token_weight(int reduction, const float* dloss, int64_t row, const int64_t* n_valid,
                                              float num_items) {
  if (reduction == 0) return __ldg(dloss + row);
  if (reduction == 1) return __ldg(dloss);
  const float den =
      num_items > 0.f ? num_items : static_cast<float>(__ldg(reinterpret_cast<const long long*>(n_valid)));
  return den > 0.f ? __ldg(dloss) / den : 0.f;
}

template <bool kBias, bool kSoftcap>
struct EpiGrad {
  using Params = GradParams;
  static constexpr int kTailBytes = kEpiSmemBytes;  // dbias column-sum staging
  __device__ static void finish(const Params&) {}
  struct State {
    int64_t row, target;
    float lse2;  // lse * log2(e)
    float w;     // per-token weight (0 for ignored tokens and rows past N)
  };

  __device__ static void begin_unit(const Params& p, const Unit& u, State& st, int /*grp*/) {
    st.row = u.row0 + epi_tid();
    st.target = p.ignore_index;
    st.lse2 = 0.f;
    st.w = 0.f;
    if (st.row < p.n_tokens) {
      st.target = __ldg(p.targets + st.row);
      st.lse2 = __ldg(p.lse + st.row) * kLog2e;
      const bool valid = st.target != p.ignore_index && st.target >= 0 && st.target < p.vocab;
      if (valid) st.w = token_weight(p.reduction, p.dloss, st.row, p.n_valid, p.num_items);
    }
  }

  // dz/dacc-weighted factor and probability of one logit (acc + bias = x).
  __device__ static void grad_terms(const Params& p, float x, float wd, float k_t, float k_p, const State& st,
                                    float& d, float& pr) {
    if (kSoftcap) {
      const float th = tanh_from_exp2_arg(x * k_t);
      pr = ex2_approx(fmaf(th, k_p, -st.lse2));          // e^(z - lse), z = c th
      d = wd * fmaf(-th, th, 1.f);                        // w s (1 - (z/c)^2)
    } else {
      pr = ex2_approx(fmaf(x, k_p, -st.lse2));            // e^(s x - lse)
      d = wd;
    }
  }

  __device__ static void tile(const Params& p, const Unit& u, int n_tile, uint32_t taddr, State& st,
                              float* epi_smem, int grp) {
    const int64_t col_tile = static_cast<int64_t>(n_tile) * kBN;  // chunk-local column
    const int64_t v_tile = p.v0 + col_tile;                       // vocabulary row
    const int warp = (threadIdx.x >> 5) & (kEpilogueWarps - 1);
    const uint32_t lane = lane_id();
    const float wd = st.w * p.scale;
    const float k_t = p.scale * p.inv_softcap * 2.0f * kLog2e;
    const float k_p = kSoftcap ? p.softcap * kLog2e : p.scale * kLog2e;
    const uint64_t k_t2 = f2_splat(k_t), k_p2 = f2_splat(k_p), nlse2 = f2_splat(-st.lse2);
    const uint64_t wd2 = f2_splat(wd), nwd2 = f2_splat(-wd);
    const uint64_t one2 = f2_splat(1.0f), mone2 = f2_splat(-1.0f), m2two2 = f2_splat(-2.0f);
    const int nch = chunks_below(v_tile, p.vocab);
    for_each_tmem_chunk<false>(taddr, nch, [&](const uint32_t (&r)[32], int c) {
      const int64_t vc = v_tile + c * 32;
      const bool ragged = vc + 32 > p.vocab;
      float bch[32];
      if (kBias) load_bias_chunk(p.bias, p.bias_f32, p.bias_vec, vc, p.vocab, bch);
      // The grad_terms arithmetic on packed fp32 pairs (columns j, j + 1); with the soft cap the
      // two columns share one reciprocal (f2_inv_exp2p1_swapped).
      float g[32];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        uint64_t x = f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
        if (kBias) x = f2_add(x, f2_pack(bch[j], bch[j + 1]));
        float q0, q1;
        if (kSoftcap) {  // from the swapped reciprocal pair on, the low lane is column j + 1
          float t0, t1;
          f2_unpack(f2_mul(x, k_t2), t0, t1);
          const uint64_t th = f2_fma(f2_inv_exp2p1_swapped(t0, t1), m2two2, one2);  // tanh
          f2_unpack(f2_fma(th, k_p2, nlse2), q0, q1);
          const uint64_t d = f2_mul(f2_fma(th, th, mone2), nwd2);  // w s (1 - th^2)
          f2_unpack(f2_mul(d, f2_pack(ex2_approx(q0), ex2_approx(q1))), g[j + 1], g[j]);
        } else {
          f2_unpack(f2_fma(x, k_p2, nlse2), q0, q1);
          f2_unpack(f2_mul(wd2, f2_pack(ex2_approx(q0), ex2_approx(q1))), g[j], g[j + 1]);
        }
      }
      const int64_t tl = st.target - vc;
      if (tl >= 0 && tl < 32) {  // the target column: subtract the one-hot term
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j == tl) {
            float x = __uint_as_float(r[j]);
            if (kBias) x += bch[j];
            float d, pr;
            grad_terms(p, x, wd, k_t, k_p, st, d, pr);
            g[j] = d * (pr - 1.f);
          }
        }
      }
      if (ragged) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (vc + j >= p.vocab) g[j] = 0.f;
      }
      if (st.row < p.n_tokens) {
        uint16_t* dst = p.g + st.row * p.ldg + col_tile + c * 32;  // 64 B, 32-byte aligned
#pragma unroll
        for (int q = 0; q < 2; ++q)
          st_global_v8(dst + 16 * q, pack_bf16x2(g[16 * q + 0], g[16 * q + 1]),
                       pack_bf16x2(g[16 * q + 2], g[16 * q + 3]), pack_bf16x2(g[16 * q + 4], g[16 * q + 5]),
                       pack_bf16x2(g[16 * q + 6], g[16 * q + 7]), pack_bf16x2(g[16 * q + 8], g[16 * q + 9]),
                       pack_bf16x2(g[16 * q + 10], g[16 * q + 11]), pack_bf16x2(g[16 * q + 12], g[16 * q + 13]),
                       pack_bf16x2(g[16 * q + 14], g[16 * q + 15]));
      }
      if (kBias && p.dbias_part) epi_smem[warp * kBN + c * 32 + lane] = warp_column_sums(g);
    });
    if (kBias && p.dbias_part) {  // (no destination with a frozen head: the bias is not trained)
      for (int c = nch; c < kBN / 32; ++c) epi_smem[warp * kBN + c * 32 + lane] = 0.f;
      epilogue_bar_sync(1 + grp);
      // A CTA-pair tile can have its second 128-row half entirely past the
      // last token: that half has no slot in the per-tile partial sums.
      if (u.row0 < p.n_tokens) {
#pragma unroll
        for (int h = 0; h < kBN / kEpilogueThreads; ++h) {
          const int col = epi_tid() + h * kEpilogueThreads;
          const float s = epi_smem[col] + epi_smem[kBN + col] + epi_smem[2 * kBN + col] + epi_smem[3 * kBN + col];
          if (v_tile + col < p.vocab) p.dbias_part[(u.row0 / kBM) * p.ldg + col_tile + col] = s;
        }
      }
      epilogue_bar_sync(1 + grp);
    }
  }

  __device__ static void end_unit(const Params&, const Unit&, State&, int) {}
};

// ============================================================================
// Epilogue: plain store (dW rows of one chunk; the test GEMM)
// ============================================================================
struct EpiStore {
  using Params = StoreParams;
  // One staging buffer per epilogue warp.
  static constexpr int kTailBytes = kEpilogueGroups * kEpilogueWarps * kStoreStageBytes;
  struct State {
    int64_t row;
  };
  __device__ static void begin_unit(const Params&, const Unit& u, State& st, int) { st.row = u.row0 + epi_tid(); }

  __device__ static void tile(const Params& p, const Unit& u, int n_tile, uint32_t taddr, State&, float* epi_smem,
                              int grp) {
    const int64_t col_tile = static_cast<int64_t>(n_tile) * kBN;
    const int nch = chunks_below(col_tile, p.cols);
    const int warp = threadIdx.x >> 5;  // 0-7: the CTA's epilogue warps
    const int64_t row_base = u.row0 + (warp % kEpilogueWarps) * 32;
    if (row_base >= p.rows) return;  // this warp's 32 rows are past the output
    uint8_t* buf = warp_stage_buffer(epi_smem, grp);
    if (p.out_f32) {  // 32 x 32 fp32 boxes (128-byte rows)
      if (u.kb_count == 0) {  // no K blocks (all tokens ignored under compaction): the product is zero
        uint32_t zero[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) zero[j] = 0u;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) store_box_tma(&p.out_map, buf, col_tile + c * 32, row_base, zero);
        return;
      }
      for_each_tmem_chunk(taddr, nch, [&](const uint32_t (&r)[32], int c) {
        store_box_tma(&p.out_map, buf, col_tile + c * 32, row_base, r);
      });
      return;
    }
    // bf16: 32 x 64 boxes, so that every row of a box is one whole 128-byte line; the two TMEM
    // chunks of a box are packed to bf16 pairs and staged like an fp32 box (128-byte rows).
#pragma unroll 1
    for (int q = 0; 2 * q < nch; ++q) {
      uint32_t w[32];
      if (u.kb_count == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = 0u;
      } else {
        const bool has_b = 2 * q + 1 < nch;
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + q * 64, ra);
        if (has_b) tmem_ld32(taddr + q * 64 + 32, rb);
        tmem_ld_wait(ra);
        if (has_b) tmem_ld_wait(rb);
        const auto f = [](uint32_t x) { return __uint_as_float(x); };
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          w[j] = pack_bf16x2(f(ra[2 * j]), f(ra[2 * j + 1]));
          w[16 + j] = has_b ? pack_bf16x2(f(rb[2 * j]), f(rb[2 * j + 1])) : 0u;
        }
      }
      store_box_tma(&p.out_map, buf, col_tile + q * 64, row_base, w);
    }
  }

  __device__ static void end_unit(const Params&, const Unit&, State&, int) {}

  __device__ static void finish(const Params&) { finish_box_stores(); }
};

// ============================================================================
// Epilogue: dh accumulation (K-split slot, or the final store)
// ============================================================================
struct EpiAccum {
  using Params = AccumParams;
  static constexpr int kTailBytes = 0;
  __device__ static void finish(const Params&) {}
  struct State {
    int64_t row;
  };
  __device__ static void begin_unit(const Params&, const Unit& u, State& st, int) { st.row = u.row0 + epi_tid(); }

  __device__ static void store(const Params& p, const Unit& u, const State& st, int64_t col, float (&v)[32]) {
    if (st.row >= p.rows) return;
    if (p.row_count && st.row >= *p.row_count) return;
    const int64_t orow = p.row_map ? static_cast<int64_t>(__ldg(p.row_map + st.row)) : st.row;
    float* slot = p.part + static_cast<int64_t>(u.ks) * p.part_stride + st.row * p.cols + col;
    const int64_t rem = p.cols - col;
    if (rem >= 32) {
      // rows are cols * 4 bytes apart (cols % 8 == 0) and col % 32 == 0: 32-byte aligned
      if (p.accumulate) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[8];
          ld_global_v8(slot + 8 * q, o);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[8 * q + i] += __uint_as_float(o[i]);
        }
      }
      const auto u = [&](int j) { return __float_as_uint(v[j]); };
      if (!p.write_final) {  // fp32 slot (32-byte aligned), read back by a later launch
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v8_cs(slot + 8 * q, u(8 * q), u(8 * q + 1), u(8 * q + 2), u(8 * q + 3), u(8 * q + 4),
                          u(8 * q + 5), u(8 * q + 6), u(8 * q + 7));
      } else if (p.out_f32) {
        float* dst = reinterpret_cast<float*>(p.out) + orow * p.cols + col;
        if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {  // the caller's output is only 16-byte aligned
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_global_v8(dst + 8 * q, u(8 * q), u(8 * q + 1), u(8 * q + 2), u(8 * q + 3), u(8 * q + 4),
                         u(8 * q + 5), u(8 * q + 6), u(8 * q + 7));
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + orow * p.cols + col;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 pk;
          pk.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
          pk.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
          pk.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
          pk.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
          reinterpret_cast<uint4*>(dst)[q] = pk;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j >= rem) continue;
        float x = v[j];
        if (p.accumulate) x += slot[j];
        if (!p.write_final) {
          slot[j] = x;
        } else if (p.out_f32) {
          reinterpret_cast<float*>(p.out)[orow * p.cols + col + j] = x;
        } else {
          reinterpret_cast<uint16_t*>(p.out)[orow * p.cols + col + j] =
              static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
        }
      }
    }
  }

  __device__ static void tile(const Params& p, const Unit& u, int n_tile, uint32_t taddr, State& st, float*,
                              int) {
    const int64_t col_tile = static_cast<int64_t>(n_tile) * kBN;
    const int nch = chunks_below(col_tile, p.cols);
    if (u.kb_count > 0) {
      for_each_tmem_chunk(taddr, nch, [&](const uint32_t (&r)[32], int c) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        store(p, u, st, col_tile + c * 32, v);
      });
    } else {  // a K split with no K blocks contributes zero
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
        store(p, u, st, col_tile + c * 32, v);
      }
    }
  }
  __device__ static void end_unit(const Params&, const Unit&, State&, int) {}
};

// ============================================================================
// The kernel
// ============================================================================
struct GemmSmem {
  uint8_t* a;          // kStages x kATileBytes
  uint8_t* b;          // kStages x kBTileBytes
  uint64_t* full;      // [kStages]  TMA -> MMA
  uint64_t* empty;     // [kStages]  MMA -> TMA
  uint64_t* tfull;     // [kAccBufs] MMA -> epilogue
  uint64_t* tempty;    // [kAccBufs] epilogue -> MMA
  uint64_t* drain;     // MMA teardown
  uint32_t* tmem_slot;
  CtaControl* ctl;
  float* epi;          // kEpiSmemBytes
};

__device__ __forceinline__ GemmSmem carve_smem(uint8_t* raw) {
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GemmSmem s;
  s.a = base;
  s.b = base + kStages * kATileBytes;
  uint8_t* bar = s.b + kStages * kBTileBytes;
  s.full = reinterpret_cast<uint64_t*>(bar);
  s.empty = s.full + kStages;
  s.tfull = s.empty + kStages;
  s.tempty = s.tfull + kAccBufs;
  s.drain = s.tempty + kAccBufs;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
  s.ctl = reinterpret_cast<CtaControl*>(s.tmem_slot + 2);
  s.epi = reinterpret_cast<float*>(bar + 1024);  // 1024-aligned epilogue region
  return s;
}

// Bounded wait used only while tearing down: waits for a copy that was issued
// to land, regardless of the abort flag.
__device__ __forceinline__ void mbar_wait_teardown(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(addr, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs / 8) return;
  }
}

// Prefetches the descriptors of the further terms that some K segment uses.
__device__ __forceinline__ void prefetch_segment_maps(const GemmSched& sc, const CUtensorMap* a1,
                                                      const CUtensorMap* a2, const CUtensorMap* b1,
                                                      const CUtensorMap* b2) {
  uint32_t used = 0;
  for (int s = 0; s < sc.nseg; ++s) {
    used |= 1u << ((sc.seg_maps >> (4 * s)) & 3u);
    used |= 16u << ((sc.seg_maps >> (4 * s + 2)) & 3u);
  }
  if (used & 2u) tma_prefetch_map(a1);
  if (used & 4u) tma_prefetch_map(a2);
  if (used & 32u) tma_prefetch_map(b1);
  if (used & 64u) tma_prefetch_map(b2);
}

template <class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                const __grid_constant__ CUtensorMap map_a2, const __grid_constant__ CUtensorMap map_b0,
                const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                const GemmSched sc, const __grid_constant__ typename Epi::Params ep, int* status) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem sm = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == kTmaWarp * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], kEpilogueWarps);
    }
    mbar_init(sm.drain, 1);
    sm.ctl->abort = 0u;
    fence_mbar_init();
    tma_prefetch_map(&map_a0);
    tma_prefetch_map(&map_b0);
    if (sc.nseg > 1) prefetch_segment_maps(sc, &map_a1, &map_a2, &map_b1, &map_b2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sm.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  // The set-up above (barriers, TMEM, descriptor prefetch) may overlap the
  // previous kernel; global memory is touched only from here on.
  griddep_wait();
  const Limits lim = read_limits(sc, kBM);

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- producer
    if (elect_one()) {
      uint32_t stage = 0, phase = 0;
      // Stages this thread has issued copies into, and the phase of the last
      // copy of each (bit masks: registers, not a local array).
      uint32_t issued = 0u, issued_phase = 0u;
      for (int uu = blockIdx.x; uu < lim.total_units; uu += gridDim.x) {
        const Unit u = decode_unit(sc, uu, kBM, 0, lim);
        if (u.skip) continue;
        bool ok = true;
        for (int n = u.n_first; ok && n < u.n_first + u.n_count; ++n) {
          for (int seg = 0; ok && seg < sc.nseg; ++seg) {
            const uint32_t ai = (sc.seg_maps >> (4 * seg)) & 3u, bi = (sc.seg_maps >> (4 * seg + 2)) & 3u;
            const CUtensorMap* ma = ai == 0 ? &map_a0 : (ai == 1 ? &map_a1 : &map_a2);
            const CUtensorMap* mb = bi == 0 ? &map_b0 : (bi == 1 ? &map_b1 : &map_b2);
            for (int kb = u.kb_first; kb < u.kb_first + u.kb_count; ++kb) {
              if (!mbar_wait(&sm.empty[stage], phase ^ 1u, sm.ctl, status)) {
                ok = false;
                break;
              }
              uint64_t* fb = &sm.full[stage];
              mbar_arrive_expect_tx(fb, kStageBytes);
              uint8_t* sa = sm.a + stage * kATileBytes;
              uint8_t* sb = sm.b + stage * kBTileBytes;
              const int k = kb * kBK;
              if (!sc.a_mn) {
                tma_load_2d(sa, ma, fb, sc.a_k_off + k, sc.a_mn_off + u.m_blk * kBM);
              } else {
#pragma unroll
                for (int j = 0; j < kBM / 64; ++j)
                  tma_load_2d(sa + j * kMnAtomBytes, ma, fb, sc.a_mn_off + u.m_blk * kBM + 64 * j, sc.a_k_off + k);
              }
              if (!sc.b_mn) {
                tma_load_2d(sb, mb, fb, sc.b_k_off + k, sc.b_mn_off + n * kBN);
              } else {
#pragma unroll
                for (int j = 0; j < kBN / 64; ++j)
                  tma_load_2d(sb + j * kMnAtomBytes, mb, fb, sc.b_mn_off + n * kBN + 64 * j, sc.b_k_off + k);
              }
              issued |= 1u << stage;
              issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
        if (!ok) break;
      }
      // Every copy this thread issued must land before the CTA may exit.
#pragma unroll
      for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u) mbar_wait_teardown(&sm.full[s], (issued_phase >> s) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (elect_one()) {
      const uint32_t idesc = instr_desc_bf16(kBM, kBN, sc.a_mn, sc.b_mn);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int uu = blockIdx.x; ok && uu < lim.total_units; uu += gridDim.x) {
        const Unit u = decode_unit(sc, uu, kBM, 0, lim);
        if (u.skip) continue;
        for (int n = u.n_first; ok && n < u.n_first + u.n_count; ++n) {
          if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, sm.ctl, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kBN;
          uint32_t accumulate = 0;
          for (int seg = 0; ok && seg < sc.nseg; ++seg) {
            for (int kb = 0; kb < u.kb_count; ++kb) {
              if (!mbar_wait(&sm.full[stage], phase, sm.ctl, status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_base = smem_u32(sm.a + stage * kATileBytes);
              const uint32_t b_base = smem_u32(sm.b + stage * kBTileBytes);
#pragma unroll
              for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                const uint64_t ad = sc.a_mn ? smem_desc_sw128(a_base + kk * 2048, kMnAtomBytes, 1024)
                                            : smem_desc_sw128(a_base + kk * 32, 16, 1024);
                const uint64_t bd = sc.b_mn ? smem_desc_sw128(b_base + kk * 2048, kMnAtomBytes, 1024)
                                            : smem_desc_sw128(b_base + kk * 32, 16, 1024);
                umma_bf16(d_tmem, ad, bd, idesc, accumulate);
                accumulate = 1;
              }
              umma_commit(&sm.empty[stage]);  // stage free once these MMAs have read it
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
          if (!ok) break;
          umma_commit(&sm.tfull[acc]);  // accumulator ready for the epilogue
          if (++acc == kAccBufs) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      // Wait for every MMA this thread issued before TMEM can be released.
      umma_commit(sm.drain);
      mbar_wait_teardown(sm.drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue (two groups)
    const int grp = warp / kEpilogueWarps;  // owns TMEM accumulator grp: tiles grp, grp+2, ...
    const uint32_t lane_base = static_cast<uint32_t>((warp % kEpilogueWarps) * 32) << 16;
    float* epi = sm.epi + grp * kEpiSmemGroupFloats;
    uint32_t seq = 0, phase = 0;
    bool ok = true;
    for (int uu = blockIdx.x; ok && uu < lim.total_units; uu += gridDim.x) {
      const Unit u = decode_unit(sc, uu, kBM, 0, lim);
        if (u.skip) continue;
      typename Epi::State st;
      Epi::begin_unit(ep, u, st, grp);
      for (int n = u.n_first; n < u.n_first + u.n_count; ++n) {
        const bool mine = static_cast<int>(seq & 1u) == grp;
        ++seq;
        if (!mine) continue;
        const bool got = mbar_wait(&sm.tfull[grp], phase, sm.ctl, status);
        if (!epilogue_all(got, 1 + grp)) {
          sm.ctl->abort = 1u;
          ok = false;
          break;
        }
        tc_fence_after();
        Epi::tile(ep, u, n, tmem_base + lane_base + grp * kBN, st, epi, grp);
        tc_fence_before();
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&sm.tempty[grp]);
        phase ^= 1u;
      }
      if (ok) Epi::end_unit(ep, u, st, grp);
    }
    Epi::finish(ep);
  }

  // The next kernel may launch once every CTA is past its work (a GEMM CTA
  // occupies its SM: dependents released earlier would only wait beside it).
  griddep_release();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}


// ============================================================================
// The CTA-pair kernel (cta_group::2): a pair of CTAs (cluster ranks 2p, 2p+1)
// computes a 256 x 256 tile.  Each CTA loads its own 128 rows of A and its own
// half of B; the pair leader's MMA thread issues M=256 MMAs that read both
// CTAs' shared memory and write 128 x 256 fp32 into each CTA's TMEM.
//   full[s]    in the leader: both CTAs' copies of stage s complete on it
//   empty[s]   in each CTA: a commit from the leader's MMA thread to each CTA
//   tfull[b]   in each CTA: a commit to each CTA, accumulator b ready
//   tempty[b]  in the leader: 4 epilogue warps of each CTA arrive (8 total)
// ============================================================================
__device__ __forceinline__ GemmSmem carve_smem_pair(uint8_t* raw) {
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GemmSmem s;
  s.a = base;
  s.b = base + kStagesPair * kATileBytes;
  uint8_t* bar = s.b + kStagesPair * kBHalfBytes;
  s.full = reinterpret_cast<uint64_t*>(bar);
  s.empty = s.full + kStagesPair;
  s.tfull = s.empty + kStagesPair;
  s.tempty = s.tfull + kAccBufs;
  s.drain = s.tempty + kAccBufs;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
  s.ctl = reinterpret_cast<CtaControl*>(s.tmem_slot + 2);
  s.epi = reinterpret_cast<float*>(bar + 1024);  // 1024-aligned epilogue region
  return s;
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

template <class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                     const __grid_constant__ CUtensorMap map_a2, const __grid_constant__ CUtensorMap map_b0,
                     const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                     const GemmSched sc, const __grid_constant__ typename Epi::Params ep, int* status) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem sm = carve_smem_pair(smem_raw);
  const int warp = threadIdx.x >> 5;
  constexpr uint32_t kCtas = 2u;
  constexpr int kTileRows = kPairRows;  // rows per unit of the pair
  const uint32_t rank = cluster_ctarank();
  const uint32_t pair_rank = rank & 1u, leader_rank = 0u;
  const bool leader = pair_rank == 0;

  if (threadIdx.x == kTmaWarp * 32) {
    for (int s = 0; s < kStagesPair; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], 2 * kEpilogueWarps);
    }
    mbar_init(sm.drain, 1);
    sm.ctl->abort = 0u;
    fence_mbar_init();
    tma_prefetch_map(&map_a0);
    tma_prefetch_map(&map_b0);
    if (sc.nseg > 1) prefetch_segment_maps(sc, &map_a1, &map_a2, &map_b1, &map_b2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(sm.tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  // The set-up above (barriers, TMEM, descriptor prefetch) may overlap the
  // previous kernel; global memory is touched only from here on.
  griddep_wait();
  const Limits lim = read_limits(sc, kTileRows);
  const int cid = static_cast<int>(blockIdx.x / kCtas);
  const int ncl = static_cast<int>(gridDim.x / kCtas);
  bool aborted = false;

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- producers (both CTAs)
    if (elect_one()) {
      uint32_t stage = 0, phase = 0;
      // Stages this thread has issued copies into, and the phase of the last
      // copy of each (bit masks: registers, not a local array).
      uint32_t issued = 0u, issued_phase = 0u;
      bool ok = true;
      for (int uu = cid; ok && uu < lim.total_units; uu += ncl) {
        const Unit u = decode_unit(sc, uu, kTileRows, rank, lim);
        if (u.skip) continue;
        const int a_row = sc.a_mn_off + static_cast<int>(u.row0);
        for (int n = u.n_first; ok && n < u.n_first + u.n_count; ++n) {
          const int b_col = sc.b_mn_off + n * kBN + static_cast<int>(pair_rank) * (kBN / 2);
          for (int seg = 0; ok && seg < sc.nseg; ++seg) {
            const uint32_t ai = (sc.seg_maps >> (4 * seg)) & 3u, bi = (sc.seg_maps >> (4 * seg + 2)) & 3u;
            const CUtensorMap* ma = ai == 0 ? &map_a0 : (ai == 1 ? &map_a1 : &map_a2);
            const CUtensorMap* mb = bi == 0 ? &map_b0 : (bi == 1 ? &map_b1 : &map_b2);
            for (int kb = u.kb_first; kb < u.kb_first + u.kb_count; ++kb) {
              if (!mbar_wait(&sm.empty[stage], phase ^ 1u, sm.ctl, status)) {
                ok = false;
                break;
              }
              const uint32_t fb = map_to_cta(smem_u32(&sm.full[stage]), leader_rank);
              if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2 * kStagePairBytes);
              uint8_t* sa = sm.a + stage * kATileBytes;
              uint8_t* sb = sm.b + stage * kBHalfBytes;
              const int k = kb * kBK;
              if (!sc.a_mn) {
                tma_load_2d_pair(sa, ma, fb, sc.a_k_off + k, a_row);
              } else {
#pragma unroll
                for (int j = 0; j < kBM / 64; ++j)
                  tma_load_2d_pair(sa + j * kMnAtomBytes, ma, fb, a_row + 64 * j, sc.a_k_off + k);
              }
              if (!sc.b_mn) {
                tma_load_2d_pair(sb, mb, fb, sc.b_k_off + k, b_col);
              } else {
#pragma unroll
                for (int j = 0; j < kBN / 128; ++j)
                  tma_load_2d_pair(sb + j * kMnAtomBytes, mb, fb, b_col + 64 * j, sc.b_k_off + k);
              }
              issued |= 1u << stage;
              issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
              if (++stage == kStagesPair) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
      }
      if (!ok) aborted = true;
      // The leader's full barriers count both CTAs' copies: wait for them to land.
      if (leader) {
#pragma unroll
        for (int s = 0; s < kStagesPair; ++s)
          if ((issued >> s) & 1u) mbar_wait_teardown(&sm.full[s], (issued_phase >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer (leader only)
    if (leader && elect_one()) {
      const uint32_t idesc = instr_desc_bf16(kPairRows, kBN, sc.a_mn, sc.b_mn);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int uu = cid; ok && uu < lim.total_units; uu += ncl) {
        const Unit u = decode_unit(sc, uu, kTileRows, rank, lim);
        if (u.skip) continue;
        for (int n = u.n_first; ok && n < u.n_first + u.n_count; ++n) {
          if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, sm.ctl, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kBN;
          uint32_t accumulate = 0;
          for (int seg = 0; ok && seg < sc.nseg; ++seg) {
            for (int kb = 0; kb < u.kb_count; ++kb) {
              if (!mbar_wait(&sm.full[stage], phase, sm.ctl, status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_base = smem_u32(sm.a + stage * kATileBytes);
              const uint32_t b_base = smem_u32(sm.b + stage * kBHalfBytes);
#pragma unroll
              for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                const uint64_t ad = sc.a_mn ? smem_desc_sw128(a_base + kk * 2048, kMnAtomBytes, 1024)
                                            : smem_desc_sw128(a_base + kk * 32, 16, 1024);
                const uint64_t bd = sc.b_mn ? smem_desc_sw128(b_base + kk * 2048, kMnAtomBytes, 1024)
                                            : smem_desc_sw128(b_base + kk * 32, 16, 1024);
                umma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
                accumulate = 1;
              }
              // stage free in both CTAs once these MMAs have read it
              const uint32_t e = smem_u32(&sm.empty[stage]);
              umma_commit_pair(e);
              umma_commit_pair(map_to_cta(e, 1u));
              if (++stage == kStagesPair) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
          if (!ok) break;
          const uint32_t tf = smem_u32(&sm.tfull[acc]);  // accumulator ready in both CTAs
          umma_commit_pair(tf);
          umma_commit_pair(map_to_cta(tf, 1u));
          if (++acc == kAccBufs) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      if (!ok) aborted = true;
      umma_commit_pair(smem_u32(sm.drain));
      mbar_wait_teardown(sm.drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs, two groups)
    const int grp = warp / kEpilogueWarps;  // owns TMEM accumulator grp: tiles grp, grp+2, ...
    const uint32_t lane_base = static_cast<uint32_t>((warp % kEpilogueWarps) * 32) << 16;
    float* epi = sm.epi + grp * kEpiSmemGroupFloats;
    uint32_t seq = 0, phase = 0;
    bool ok = true;
    for (int uu = cid; ok && uu < lim.total_units; uu += ncl) {
      const Unit u = decode_unit(sc, uu, kTileRows, rank, lim);
        if (u.skip) continue;
      typename Epi::State st;
      Epi::begin_unit(ep, u, st, grp);
      for (int n = u.n_first; n < u.n_first + u.n_count; ++n) {
        const bool mine = static_cast<int>(seq & 1u) == grp;
        ++seq;
        if (!mine) continue;
        const bool got = mbar_wait(&sm.tfull[grp], phase, sm.ctl, status);
        if (!epilogue_all(got, 1 + grp)) {
          sm.ctl->abort = 1u;
          ok = false;
          break;
        }
        tc_fence_after();
        Epi::tile(ep, u, n, tmem_base + lane_base + grp * kBN, st, epi, grp);
        tc_fence_before();
        __syncwarp();
        if (lane_id() == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&sm.tempty[grp]), leader_rank));
        phase ^= 1u;
      }
      if (ok) Epi::end_unit(ep, u, st, grp);
    }
    Epi::finish(ep);
    if (!ok) aborted = true;
  }

  // The next kernel may launch once every CTA is past its work (a GEMM CTA
  // occupies its SM: dependents released earlier would only wait beside it).
  griddep_release();
  // After an abort, copies the other CTA issued may still be in flight toward
  // this CTA's shared memory or barriers: give them time to land.
  if (aborted || sm.ctl->abort) spin_ns(100000);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace flce
