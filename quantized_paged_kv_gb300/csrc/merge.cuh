// merge.cuh — the log-sum-exp combine of split partials: the task code of the
// merge kernel (its warp count and CTA barrier are parameters)
// ("long-context-attention-and-lessons", section "Give more GPU workers a piece
// of the attention calculation": each piece produces a weighted value sum and the
// information needed to normalise it; averaging the partial outputs would be
// incorrect).
//
//   M = max_s lse_s,  w_s = exp(lse_s - M),  out = sum_s w_s o_s / sum_s w_s,
//   lse = M + log(sum_s w_s);  a split with lse = -inf (no tokens) has weight 0.
//
// Work unit: a task = (sequence, query head, slice of D columns), merged by WPR
// warps.  Within a warp, L = 32 / R lanes cover the slice (4 columns each, float4)
// and the R lane phases take different splits, so one load instruction brings R
// partial rows; each lane keeps eight loads in flight.  The shape is the same for
// the whole launch and is chosen on the device from the largest split count of
// the batch (every CTA scans the split offsets first):
//   * at most 16 splits: R = 1 (128-column slices), WPR = 1 — one task per warp;
//   * more: R = 4 (32-column slices) and WPR up to the CTA's warp count, so a
//     long sequence's rows spread over many CTAs and each CTA still has many
//     rows in flight.
// Each lane keeps a running maximum of the lse values it has seen and rescales
// its sums when it grows (one pass over the partials); lane phases and warps are
// then combined the same way (by shuffles, and through shared memory).
// Sequences with a single split are skipped (the decode kernel wrote them).
// Split offsets come from the plan, or (offs = null) every sequence has
// `uniform` splits at rows b * uniform ...  CTAs
// walk groups of NW / WPR tasks, grid-stride.  Partials are read with L1 bypassed
// (they were written by other SMs).
#pragma once

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

constexpr int kMinSliceCols = 32;  // narrowest slice (R = 4)
constexpr int kShortSplits = 16;   // up to this many splits: R = 1, WPR = 1
constexpr int kInFlight = 8;       // loads in flight per lane

template <int R, int NW, class Sync>
__device__ __forceinline__ void merge_tasks(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                            const int32_t* __restrict__ offs, int uniform, int batch, int num_q_heads, int D,
                                            void* out, int out_bf16, float* lse_out, int wpr,
                                            float4 (*red_o)[32], float* red_w, float* red_m, Sync sync) {
  constexpr int L = 32 / R;            // lanes per row
  constexpr int kCols = 4 * L;         // columns per task
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int phase = lane / L, col = lane % L;
  const int tasks_per_group = NW / wpr;
  const int sub = warp % wpr;
  const int slot = warp / wpr;
  const int slices = D / kCols;
  const int64_t tasks = (int64_t)batch * num_q_heads * slices;
  const int64_t groups = (tasks + tasks_per_group - 1) / tasks_per_group;
  const size_t ostride = (size_t)num_q_heads * D;
  const int row0 = sub * R + phase;     // first split of this lane
  const int rstep = wpr * R;            // splits between this lane's rows
  for (int64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int64_t t = grp * tasks_per_group + slot;
    int S = 0, base = 0, b = 0, g = 0, slice = 0;
    if (t < tasks) {
      const int bg = static_cast<int>(t / slices);
      slice = static_cast<int>(t - (int64_t)bg * slices);
      b = bg / num_q_heads;
      g = bg - b * num_q_heads;
      base = offs ? offs[b] : b * uniform;
      S = offs ? offs[b + 1] - base : uniform;
    }
    // one pass with an online rescale: (m, wsum, acc) = running max of the lse
    // values seen, sum of exp(lse - m), and sum of exp(lse - m) * o
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f, m = -INFINITY;
    const bool active = S > 1;  // uniform over the task's warps
    if (active) {
      const float* lrow = lse_part + (size_t)base * num_q_heads + g;  // stride num_q_heads
      const float* orow = o_part + (size_t)base * ostride + (size_t)g * D + slice * kCols + col * 4;
      for (int s0 = row0; s0 < S; s0 += kInFlight * rstep) {
        float l[kInFlight];
        float4 v[kInFlight];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
          const int s = s0 + u * rstep;
          l[u] = -INFINITY;
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (s < S) {
            l[u] = __ldcg(lrow + (size_t)s * num_q_heads);
            v[u] = __ldcg(reinterpret_cast<const float4*>(orow + (size_t)s * ostride));
          }
        }
        float lm = m;
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) lm = fmaxf(lm, l[u]);
        if (lm != -INFINITY) {
          const float sc = expf(m - lm);  // m = -inf: 0 (acc and wsum are 0 then)
          wsum *= sc;
          acc.x *= sc;
          acc.y *= sc;
          acc.z *= sc;
          acc.w *= sc;
          m = lm;
#pragma unroll
          for (int u = 0; u < kInFlight; ++u) {
            const float w = l[u] == -INFINITY ? 0.f : expf(l[u] - m);
            wsum += w;
            acc.x += w * v[u].x;
            acc.y += w * v[u].y;
            acc.z += w * v[u].z;
            acc.w += w * v[u].w;
          }
        }
      }
#pragma unroll
      for (int o = L; o < 32; o <<= 1) {  // combine the lane phases
        const float mo = __shfl_xor_sync(0xffffffffu, m, o);
        const float wo = __shfl_xor_sync(0xffffffffu, wsum, o);
        const float ax = __shfl_xor_sync(0xffffffffu, acc.x, o);
        const float ay = __shfl_xor_sync(0xffffffffu, acc.y, o);
        const float az = __shfl_xor_sync(0xffffffffu, acc.z, o);
        const float aw = __shfl_xor_sync(0xffffffffu, acc.w, o);
        const float mn = fmaxf(m, mo);
        const float s1 = mn == -INFINITY ? 0.f : expf(m - mn), s2 = mn == -INFINITY ? 0.f : expf(mo - mn);
        wsum = wsum * s1 + wo * s2;
        acc.x = acc.x * s1 + ax * s2;
        acc.y = acc.y * s1 + ay * s2;
        acc.z = acc.z * s1 + az * s2;
        acc.w = acc.w * s1 + aw * s2;
        m = mn;
      }
    }
    if (wpr > 1) {  // combine the task's warps (uniform branch)
      red_o[warp][lane] = acc;
      if (lane == 0) {
        red_w[warp] = wsum;
        red_m[warp] = m;
      }
      sync();
      if (sub == 0) {
        float mn = m;
        for (int j = 1; j < wpr; ++j) mn = fmaxf(mn, red_m[warp + j]);
        const float s0 = mn == -INFINITY ? 0.f : expf(m - mn);
        wsum *= s0;
        acc.x *= s0;
        acc.y *= s0;
        acc.z *= s0;
        acc.w *= s0;
        for (int j = 1; j < wpr; ++j) {
          const float sj = mn == -INFINITY ? 0.f : expf(red_m[warp + j] - mn);
          const float4 v = red_o[warp + j][lane];
          acc.x += v.x * sj;
          acc.y += v.y * sj;
          acc.z += v.z * sj;
          acc.w += v.w * sj;
          wsum += red_w[warp + j] * sj;
        }
        m = mn;
      }
      sync();  // the buffers are reused by the next group
    }
    if (active && sub == 0 && phase == 0) {
      float lse = -INFINITY;
      if (m != -INFINITY && wsum > 0.f) {
        const float inv = 1.f / wsum;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        lse = m + logf(wsum);
      } else {
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const size_t off = ((size_t)b * num_q_heads + g) * D + slice * kCols + col * 4;
      if (out_bf16) {
        __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(out) + off);
        ob[0] = __floats2bfloat162_rn(acc.x, acc.y);
        ob[1] = __floats2bfloat162_rn(acc.z, acc.w);
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + off) = acc;
      }
      if (slice == 0 && col == 0 && lse_out) lse_out[(size_t)b * num_q_heads + g] = lse;
    }
  }
}


// Largest split count of the batch (every thread of the NW warps gets it).
template <int NW, class Sync>
__device__ __forceinline__ int merge_max_splits(const int32_t* __restrict__ offs, int uniform, int batch, int* red_s,
                                                Sync sync) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int smax = 0;
  if (!offs) return uniform;
  for (int b = tid; b < batch; b += NW * 32) smax = max(smax, offs[b + 1] - offs[b]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, o));
  if (lane == 0) red_s[warp] = smax;
  sync();
  smax = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) smax = max(smax, red_s[w]);
  return smax;
}

// All merge tasks of the batch for a grid of CTAs with NW warps each (threads
// 0 .. NW*32-1 of the CTA take part); smax = merge_max_splits(...).
template <int NW, class Sync>
__device__ __forceinline__ void merge_all(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                          const int32_t* __restrict__ offs, int uniform, int batch, int num_q_heads, int D,
                                          void* out, int out_bf16, float* lse_out, int smax,
                                          float4 (*red_o)[32], float* red_w, float* red_m, Sync sync) {
  if (smax <= 1) return;  // nothing to merge
  if (smax <= kShortSplits) {
    merge_tasks<1, NW>(o_part, lse_part, offs, uniform, batch, num_q_heads, D, out, out_bf16, lse_out, 1, red_o, red_w, red_m,
                       sync);
  } else {
    int wpr = 1;  // 4 splits per warp-load, 8 loads in flight: 32 splits per warp per round
    while (wpr < NW && (NW % (2 * wpr)) == 0 && wpr * 4 * kInFlight < smax) wpr <<= 1;
    merge_tasks<4, NW>(o_part, lse_part, offs, uniform, batch, num_q_heads, D, out, out_bf16, lse_out, wpr, red_o, red_w, red_m,
                       sync);
  }
}

}  // namespace kvq
