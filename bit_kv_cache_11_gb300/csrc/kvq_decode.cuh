// kvq_decode.cuh — split-K decode attention over the packed cache (template).
//
// Attention output = softmax-weighted sum of value vectors ("Your KV cache
// doesn't have a bit problem, it has a geometry problem", section "Values:
// Where the Intuition Breaks"); keys stored before RoPE are rotated after
// dequantization (section "Rotary Embeddings Complicate the Keys"); the GPU
// reads the whole cache once per generated token (section "Why the KV Cache
// Is Where This Bites"), so the kernel is built to stream HBM.
//
// Work decomposition.  Units are (pair, 32-token sub-block) plus one fp16
// unit per pair for the tail and one for the sink window (when present); warp
// w of the grid owns a contiguous range of units (kvq_device.cuh, UnitMap: an
// equal share of the cost, where every pair adds a few virtual units for the
// work of leaving it), so every warp streams contiguous memory and all warps
// get the same amount of work whatever the batch/head/context shape.  A warp keeps
// one online-softmax state (m, l, o) per query head of the GQA group and
// writes it as a partial for every pair its range touches; the merge kernel
// combines the partials of a pair.
//
// Data movement.  Each warp owns NS shared-memory stages.  Lane 0 issues the
// one-dimensional TMA bulk copies (K codes, K metadata, V codes, V metadata)
// of a sub-block into a stage and arms the stage's mbarrier with the byte
// count; the warp waits on the barrier (bounded), computes, and refills the
// stage with the sub-block NS units ahead.
//
// Arithmetic per sub-block (lane j = token j):
//   channel-axis keys:  q.k_j = sum_d (q_d s_d) c_jd + sum_d q_d z_d — the
//                       scale is folded into the query once per sub-block;
//   token-axis keys:    q.k_j = sum_g s_jg sum_{d in g} q_d c_jd + z_jg sum_{d in g} q_d;
//   RoPE keys:          k_jd = fma(c, s, z), rotated at the token's position;
//   token-axis values:  o_d += (p_j s_jg) c_jd  and  Z_g += p_j z_jg;
//   channel-axis values: o_d += s_d sum_j p_j c_jd + z_d sum_j p_j.
// Scores are kept in log2 units (the query is pre-multiplied by scale*log2 e).
#pragma once

#include "kvq_device.cuh"

namespace kvq {

constexpr int kDecodeWarps = 4;

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int BK, int BV, int R>
struct DecodeCfg {
  static constexpr int KW = D * BK / 32;  // words per K row
  static constexpr int CPL = D / 32;      // value channels per lane
  static constexpr int KC_S = 4 * D * BK; // 32 tokens x D x BK bits
  static constexpr int KM_S = 4 * D;
  static constexpr int VC_S = 4 * D * BV;
  static constexpr int VM_S = 4 * D;
  static constexpr int STAGE = KC_S + KM_S + VC_S + VM_S;
  static constexpr int NS = STAGE <= 4096 ? 4 : (STAGE <= 10240 ? 3 : 2);
  static constexpr int OFF_BAR = NS * STAGE;
  static constexpr int OFF_QS = OFF_BAR + 64;
  static constexpr int OFF_QT = OFF_QS + R * D * 4;
  static constexpr int OFF_PB = OFF_QT + R * D * 4;
  static constexpr int OFF_QG = OFF_PB + R * 32 * 4;
  static constexpr int WARP_BYTES = round_up(OFF_QG + R * 4 * 4, 128);
  static constexpr int SMEM = kDecodeWarps * WARP_BYTES;
  static_assert(KW % 4 == 0, "K rows are read as 16-byte vectors");
  static_assert((CPL * BV) % 2 == 0, "V words are read in pairs");
};

template <int D, int BK, int BV, int R, bool F8 = false>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_split_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, BK, BV, R>;
  constexpr int NS = C::NS;
  constexpr uint32_t KMASK = (1u << BK) - 1u;
  constexpr uint32_t VMASK = (1u << BV) - 1u;
  constexpr int KPER = 32 / BK;
  constexpr int VPER = 32 / BV;
  constexpr int CPL = C::CPL;

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * kDecodeWarps + warp;
  if (gw >= p.n_warps) return;

  uint8_t* ws = smem + warp * C::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ws + C::OFF_BAR);
  float* qs = reinterpret_cast<float*>(ws + C::OFF_QS);  // [R][D] scaled query
  float* qt = reinterpret_cast<float*>(ws + C::OFF_QT);  // [R][D] query * key scale
  float* pb = reinterpret_cast<float*>(ws + C::OFF_PB);  // [R][32] probabilities
  float* qg = reinterpret_cast<float*>(ws + C::OFF_QG);  // [R][4] per-group query sums

  const int G = p.g.G;
  const int lgG = p.lg_G;
  const int ng = D >> lgG;     // channel groups per token (token axis); 0 if G > D
  const int sub_mask = (1 << p.lg_sub) - 1;
  int ua_i, ub_i;
  warp_units(p.map, static_cast<int>(gw), &ua_i, &ub_i);
  const long long ua = ua_i, ub = ub_i;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Load cursor: the next quantized unit to copy (fp16 units are skipped).
  UnitCursor lc;
  lc.init(p, ua, ub);
  auto skip_tail = [&]() {
    while (lc.u < ub && lc.j >= lc.l.nsub) lc.next(p);
  };
  UnitCursor uc;  // the compute cursor
  uc.init(p, ua, ub);
  // Lane 0: copies of quantized unit u into stage s.
  auto issue = [&](long long pr, int j, int s) {
    const int blk = j >> p.lg_sub;
    const int ch = j & sub_mask;
    const uint8_t* base =
        p.g.blocks + (static_cast<size_t>(pr) * p.g.NB + blk) * p.g.block_bytes;
    uint8_t* st = ws + s * C::STAGE;
    const uint32_t km_bytes = p.g.ak == 0 ? 4u * D : 128u * ng;
    const uint32_t vm_bytes = p.g.av == 0 ? 4u * D : 128u * ng;
    const uint8_t* km_src = base + p.g.off_km + (p.g.ak == 0 ? 0 : ch * 128 * ng);
    const uint8_t* vm_src = base + p.g.off_vm + (p.g.av == 0 ? 0 : ch * 128 * ng);
    mbar_arrive_expect_tx(&bars[s], C::KC_S + km_bytes + C::VC_S + vm_bytes);
    bulk_g2s(st, base + ch * C::KC_S, C::KC_S, &bars[s]);
    bulk_g2s(st + C::KC_S, km_src, km_bytes, &bars[s]);
    bulk_g2s(st + C::KC_S + C::KM_S, base + p.g.off_vc + ch * C::VC_S, C::VC_S, &bars[s]);
    bulk_g2s(st + C::KC_S + C::KM_S + C::VC_S, vm_src, vm_bytes, &bars[s]);
  };

  skip_tail();
  int issued = 0;
  for (int s = 0; s < NS && lc.u < ub; ++s) {
    if (lane == 0) issue(lc.pr, lc.j, s);
    ++issued;
    lc.next(p);
    skip_tail();
  }

  float m[R], l[R], zacc[R];
  float acc[R][CPL];
  long long cur = -1;
  int qi = 0;

  auto enter_pair = [&](long long pr) {
    const __half* qp = p.q + static_cast<size_t>(pr) * R * D;
    for (int i = lane; i < R * D; i += 32) qs[i] = __half2float(qp[i]) * p.qscale;
    __syncwarp();
    if (p.g.ak == 1 && lane < R * ng) {
      const int r = lane / ng, g = lane % ng;
      float sum = 0.f;
      for (int d = g * G; d < (g + 1) * G; ++d) sum += qs[r * D + d];
      qg[r * 4 + g] = sum;
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
      zacc[r] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[r][c] = 0.f;
    }
  };

  auto write_partial = [&](long long pr) {
    const long long slot = gw + pr;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (lane == 0) p.part_ml[slot * R + r] = make_float2(m[r], l[r]);
      float* o = p.part_o + (slot * R + r) * D + lane * CPL;
#pragma unroll
      for (int c = 0; c < CPL; ++c) o[c] = acc[r][c] + zacc[r];
    }
  };

  // Online softmax over the 32 lanes' scores; leaves p_j in pb.
  auto softmax_update = [&](float (&sc)[R], float (&psum)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float mx = warp_max(sc[r]);
      const float mn = fmaxf(m[r], mx);
      const float alpha = exp2f(m[r] - mn);
      const float pj = exp2f(sc[r] - mn);
      psum[r] = warp_sum(pj);
      l[r] = l[r] * alpha + psum[r];
      m[r] = mn;
      zacc[r] *= alpha;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[r][c] *= alpha;
      pb[r * 32 + lane] = pj;
    }
    __syncwarp();
  };

  auto process_sub = [&](const uint8_t* st, int j) {
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st);
    const __half2* km = reinterpret_cast<const __half2*>(st + C::KC_S);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + C::KC_S + C::KM_S);
    const __half2* vm = reinterpret_cast<const __half2*>(st + C::KC_S + C::KM_S + C::VC_S);
    float sc[R];
    // ---- scores, lane = token
    uint32_t kr[C::KW];
    {
      const uint4* row = reinterpret_cast<const uint4*>(kc + lane * C::KW);
#pragma unroll
      for (int v = 0; v < C::KW / 4; ++v) {
        const uint4 w4 = row[v];
        kr[4 * v + 0] = w4.x;
        kr[4 * v + 1] = w4.y;
        kr[4 * v + 2] = w4.z;
        kr[4 * v + 3] = w4.w;
      }
    }
    auto kcode = [&](int d) -> float {
      return code_value<F8>((kr[d / KPER] >> ((d % KPER) * BK)) & KMASK);
    };
    if (p.rope) {
      const int pos = uc.l.Ts + j * 32 + lane;
      const float2* cs = p.rope_tab + static_cast<size_t>(pos) * (D / 2);
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = 0.f;
#pragma unroll
      for (int i = 0; i < D / 2; ++i) {
        const int i1 = i + D / 2;
        const float2 m0 = __half22float2(km[p.g.ak == 0 ? i : lane * ng + (i >> lgG)]);
        const float2 m1 = __half22float2(km[p.g.ak == 0 ? i1 : lane * ng + (i1 >> lgG)]);
        const float k0 = fmaf(kcode(i), m0.x, m0.y);
        const float k1 = fmaf(kcode(i1), m1.x, m1.y);
        const float2 t = cs[i];
        const float r0 = k0 * t.x - k1 * t.y;
        const float r1 = k1 * t.x + k0 * t.y;
#pragma unroll
        for (int r = 0; r < R; ++r) sc[r] += qs[r * D + i] * r0 + qs[r * D + i1] * r1;
      }
    } else if (p.g.ak == 0) {
      float cz[R];
#pragma unroll
      for (int r = 0; r < R; ++r) cz[r] = 0.f;
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        const int d = lane + 32 * k;
        const float2 sz = __half22float2(km[d]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float v = qs[r * D + d];
          qt[r * D + d] = v * sz.x;
          cz[r] = fmaf(v, sz.y, cz[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = warp_sum(cz[r]);
      __syncwarp();
#pragma unroll
      for (int d = 0; d < D; d += 4) {
        const float c0 = kcode(d), c1 = kcode(d + 1), c2 = kcode(d + 2), c3 = kcode(d + 3);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 w = *reinterpret_cast<const float4*>(qt + r * D + d);
          sc[r] = fmaf(w.x, c0, sc[r]);
          sc[r] = fmaf(w.y, c1, sc[r]);
          sc[r] = fmaf(w.z, c2, sc[r]);
          sc[r] = fmaf(w.w, c3, sc[r]);
        }
      }
    } else {
      float part[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        sc[r] = 0.f;
        part[r] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
#pragma unroll
        for (int d = 32 * k; d < 32 * k + 32; d += 4) {
          const float c0 = kcode(d), c1 = kcode(d + 1), c2 = kcode(d + 2), c3 = kcode(d + 3);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float4 w = *reinterpret_cast<const float4*>(qs + r * D + d);
            part[r] = fmaf(w.x, c0, part[r]);
            part[r] = fmaf(w.y, c1, part[r]);
            part[r] = fmaf(w.z, c2, part[r]);
            part[r] = fmaf(w.w, c3, part[r]);
          }
        }
        if ((((k + 1) * 32) & (G - 1)) == 0) {  // a channel group closes
          const int g = (k * 32) >> lgG;
          const float2 sz = __half22float2(km[lane * ng + g]);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            sc[r] += sz.x * part[r] + sz.y * qg[r * 4 + g];
            part[r] = 0.f;
          }
        }
      }
    }
    float psum[R];
    softmax_update(sc, psum);

    // ---- values, lane = channels [lane*CPL, +CPL)
    const int d0 = lane * CPL;
    uint32_t vw[CPL * BV];
    {
      const uint2* src = reinterpret_cast<const uint2*>(vc + d0 * BV);
#pragma unroll
      for (int v = 0; v < CPL * BV / 2; ++v) {
        const uint2 w2 = src[v];
        vw[2 * v] = w2.x;
        vw[2 * v + 1] = w2.y;
      }
    }
    if (p.g.av == 1) {
      const int g = d0 >> lgG;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const float2 sz = __half22float2(vm[t * ng + g]);
        const int w = t / VPER, sh = (t % VPER) * BV;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pr = pb[r * 32 + t];
          const float pt = pr * sz.x;
          zacc[r] = fmaf(pr, sz.y, zacc[r]);
#pragma unroll
          for (int c = 0; c < CPL; ++c)
            acc[r][c] = fmaf(pt, code_value<F8>((vw[c * BV + w] >> sh) & VMASK), acc[r][c]);
        }
      }
    } else {
      float a[R][CPL];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) a[r][c] = 0.f;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int w = t / VPER, sh = (t % VPER) * BV;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pr = pb[r * 32 + t];
#pragma unroll
          for (int c = 0; c < CPL; ++c)
            a[r][c] = fmaf(pr, code_value<F8>((vw[c * BV + w] >> sh) & VMASK), a[r][c]);
        }
      }
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float2 sz = __half22float2(vm[d0 + c]);
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r][c] += sz.x * a[r][c] + sz.y * psum[r];
      }
    }
    __syncwarp();
  };

  // fp16 rows [0, nrows) of kt / vt (the tail, or the sink window), row t
  // at position pos0 + t.
  auto process_rows = [&](const __half* kt, const __half* vt, int nrows, int pos0) {
    const int d0 = lane * CPL;
    for (int t0 = 0; t0 < nrows; t0 += 32) {
      const int t = t0 + lane;
      float sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = 0.f;
      if (t < nrows) {
        const __half* row = kt + static_cast<size_t>(t) * D;
        if (p.rope) {
          const float2* cs = p.rope_tab + static_cast<size_t>(pos0 + t) * (D / 2);
          for (int i = 0; i < D / 2; i += 8) {
            const uint4 a4 = *reinterpret_cast<const uint4*>(row + i);
            const uint4 b4 = *reinterpret_cast<const uint4*>(row + i + D / 2);
            const __half2* a2 = reinterpret_cast<const __half2*>(&a4);
            const __half2* b2 = reinterpret_cast<const __half2*>(&b4);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float k0 = __half2float(e % 2 == 0 ? a2[e / 2].x : a2[e / 2].y);
              const float k1 = __half2float(e % 2 == 0 ? b2[e / 2].x : b2[e / 2].y);
              const float2 cs2 = cs[i + e];
              const float r0 = k0 * cs2.x - k1 * cs2.y;
              const float r1 = k1 * cs2.x + k0 * cs2.y;
#pragma unroll
              for (int r = 0; r < R; ++r)
                sc[r] += qs[r * D + i + e] * r0 + qs[r * D + i + e + D / 2] * r1;
            }
          }
        } else {
          for (int d = 0; d < D; d += 8) {
            const uint4 a4 = *reinterpret_cast<const uint4*>(row + d);
            const __half2* a2 = reinterpret_cast<const __half2*>(&a4);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kk = __half22float2(a2[e]);
#pragma unroll
              for (int r = 0; r < R; ++r) {
                sc[r] = fmaf(qs[r * D + d + 2 * e], kk.x, sc[r]);
                sc[r] = fmaf(qs[r * D + d + 2 * e + 1], kk.y, sc[r]);
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) sc[r] = -INFINITY;
      }
      float psum[R];
      softmax_update(sc, psum);
      const int nt = min(32, nrows - t0);
      for (int jj = 0; jj < nt; ++jj) {
        const __half* vr = vt + static_cast<size_t>(t0 + jj) * D + d0;
        float vv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) vv[c] = __half2float(vr[c]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pr = pb[r * 32 + jj];
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[r][c] = fmaf(pr, vv[c], acc[r][c]);
        }
      }
      __syncwarp();
    }
  };

  for (; uc.u < ub; uc.next(p)) {
    const long long pr = uc.pr;
    const int j = uc.j;
    if (pr != cur) {
      if (cur >= 0) write_partial(cur);
      enter_pair(pr);
      cur = pr;
    }
    if (j >= uc.l.nsub) {
      const PairLens& l = uc.l;
      if (j < l.nsub + l.ntu)
        process_rows(p.ktail[l.buf] + static_cast<size_t>(pr) * p.g.TC * D,
                     p.vtail[l.buf] + static_cast<size_t>(pr) * p.g.TC * D, l.Tt, l.Ts + l.Tq);
      else
        process_rows(p.ksink + static_cast<size_t>(pr) * p.g.NSK * D,
                     p.vsink + static_cast<size_t>(pr) * p.g.NSK * D, l.Ts, 0);
      continue;
    }
    const int s = qi % NS;
    if (!mbar_wait_bounded(&bars[s], static_cast<uint32_t>((qi / NS) & 1), p.wait_limit)) {
      // Give up: record the error, wait (bounded) for this warp's copies in
      // flight so no bulk copy lands after the CTA exits, and return.
      if (lane == 0) atomicExch(p.err, kDevErrWait);
      for (int k = qi; k < issued; ++k)
        mbar_wait_bounded(&bars[k % NS], static_cast<uint32_t>((k / NS) & 1));
      return;
    }
    process_sub(ws + s * C::STAGE, j);
    ++qi;
    if (lc.u < ub) {
      if (lane == 0) issue(lc.pr, lc.j, s);
      ++issued;
      lc.next(p);
      skip_tail();
    }
  }
  if (cur >= 0) write_partial(cur);
}

// Host-side entry points of one instantiation.
template <int D, int BK, int BV, int R, bool F8 = false>
cudaError_t decode_prepare(int* warps_per_sm) {
  using C = DecodeCfg<D, BK, BV, R>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, BK, BV, R, F8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int ctas = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &ctas, decode_split_kernel<D, BK, BV, R, F8>, kDecodeWarps * 32, C::SMEM);
  *warps_per_sm = ctas * kDecodeWarps;
  return e;
}

template <int D, int BK, int BV, int R, bool F8 = false>
cudaError_t decode_launch(const DecodeParams& p, cudaStream_t stream) {
  using C = DecodeCfg<D, BK, BV, R>;
  const int grid = (p.n_warps + kDecodeWarps - 1) / kDecodeWarps;
  decode_split_kernel<D, BK, BV, R, F8><<<grid, kDecodeWarps * 32, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

struct DecodeOps {
  cudaError_t (*prepare)(int* warps_per_sm);  // opt-ins; resident warps per SM
  cudaError_t (*launch)(const DecodeParams& p, cudaStream_t stream);
};

template <int D, int R>
DecodeOps decode_ops_for(int bk, int bv) {
#define KVQ_CASE(BK_, BV_) \
  if (bk == BK_ && bv == BV_) return DecodeOps{decode_prepare<D, BK_, BV_, R>, decode_launch<D, BK_, BV_, R>};
  KVQ_CASE(2, 2) KVQ_CASE(2, 4) KVQ_CASE(2, 8)
  KVQ_CASE(4, 2) KVQ_CASE(4, 4) KVQ_CASE(4, 8)
  KVQ_CASE(8, 2) KVQ_CASE(8, 4) KVQ_CASE(8, 8)
#undef KVQ_CASE
  if (bk == kBitsE4M3 && bv == kBitsE4M3)
    return DecodeOps{decode_prepare<D, 8, 8, R, true>, decode_launch<D, 8, 8, R, true>};
  return DecodeOps{nullptr, nullptr};
}

// Defined in the per-(D, R) translation units.
DecodeOps decode_ops(int D, int R, int bk, int bv);

}  // namespace kvq
