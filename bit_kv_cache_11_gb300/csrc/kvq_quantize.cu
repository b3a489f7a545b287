// kvq_quantize.cu — prefill quantization, decode-time append with the tail
// flush, and the dequantize test path.
//
// The quantizer ("Your KV cache doesn't have a bit problem, it has a geometry
// problem", section "What Quantization Error Is Actually Made Of"): per group
// zero point = minimum, step = (max - min) / (2^B - 1), round each element to
// the nearest step.  Keys are grouped per channel over G tokens and values
// per token over G channels (sections "Keys: The Outliers Live in Fixed
// Channels", "Values: Where the Intuition Breaks"); both axes are selectable.
// The fp16 tail and its flush in whole groups follow section "The Systems
// Tax, and Why It Is Not a Detail".
//
// One CTA quantizes one G-token block of one (batch, kv-head) pair:
//   1. 16-byte loads of the block's G fp16 K rows and V rows into shared
//      memory (the rows come from the old tail or the new tokens);
//   2. per group min/max -> fp32 step -> fp16 {scale, zero} metadata;
//   3. codes packed into uint32 words, one word per thread, written with
//      coalesced stores in the block layout of include/kvq.h.
// The extra CTA x == nflush copies the remainder tokens into the tail.
#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kQuantThreads = 256;

struct Stat {
  float mn;
  float s;  // fp32 value of the stored fp16 step
};

// Group statistics of n values x[0], x[stride], ...: writes the fp16 metadata
// and returns the fp32 minimum and stored step used for the codes.
__device__ __forceinline__ Stat group_stat(const __half* x, int stride, int n, int bits,
                                           __half2* meta_out) {
  float mn = __half2float(x[0]);
  float mx = mn;
  for (int i = 1; i < n; ++i) {
    float v = __half2float(x[i * stride]);
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
  // (mx - mn) + 0: a range of -0 (min and max zeros of opposite sign) is +0.
  float range = __fadd_rn(__fsub_rn(mx, mn), 0.0f);
  float step = __fdiv_rn(range, static_cast<float>((1 << bits) - 1));
  __half s_h = __float2half_rn(step);
  __half z_h = __float2half_rn(__fadd_rn(mn, 0.0f));  // a -0 minimum is stored as +0
  *meta_out = __halves2half2(s_h, z_h);
  return Stat{mn, __half2float(s_h)};
}

__device__ __forceinline__ uint32_t code_of(float x, Stat st, int bits) {
  if (st.s == 0.0f) return 0u;
  float r = rintf(__fdiv_rn(__fsub_rn(x, st.mn), st.s));
  r = fminf(fmaxf(r, 0.0f), static_cast<float>((1 << bits) - 1));
  return static_cast<uint32_t>(r);
}

__device__ __forceinline__ const __half* combined_row(const QuantParams& q, int p, int jc) {
  const int D = q.g.D;
  if (jc < q.T_t) return q.kold + (static_cast<size_t>(p) * q.g.G + jc) * D;
  return q.knew + (static_cast<size_t>(p) * q.n + (jc - q.T_t)) * D;
}

__device__ __forceinline__ const __half* combined_row_v(const QuantParams& q, int p, int jc) {
  const int D = q.g.D;
  if (jc < q.T_t) return q.vold + (static_cast<size_t>(p) * q.g.G + jc) * D;
  return q.vnew + (static_cast<size_t>(p) * q.n + (jc - q.T_t)) * D;
}

}  // namespace

__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const QuantParams q) {
  const int x = blockIdx.x;
  const int p = blockIdx.y;
  const int D = q.g.D, G = q.g.G;
  const int tid = threadIdx.x;

  if (x == q.nflush) {
    // remainder -> tail rows [dst_row0, ...)
    const int rows = q.rem_end - q.rem_begin;
    const int chunks = rows * (D / 8);
    for (int c = tid; c < chunks; c += blockDim.x) {
      const int r = c / (D / 8);
      const int col = (c % (D / 8)) * 8;
      const int jc = q.rem_begin + r;
      const size_t dst = (static_cast<size_t>(p) * G + q.dst_row0 + r) * D + col;
      *reinterpret_cast<uint4*>(q.kdst + dst) =
          *reinterpret_cast<const uint4*>(combined_row(q, p, jc) + col);
      *reinterpret_cast<uint4*>(q.vdst + dst) =
          *reinterpret_cast<const uint4*>(combined_row_v(q, p, jc) + col);
    }
    return;
  }

  extern __shared__ __align__(16) uint8_t smem[];
  __half* xk = reinterpret_cast<__half*>(smem);
  __half* xv = xk + G * D;
  Stat* sk = reinterpret_cast<Stat*>(xv + G * D);
  Stat* sv = sk + D;

  // 1. load the block's rows (combined index x*G + j)
  const int chunks = G * (D / 8);
  for (int c = tid; c < chunks; c += blockDim.x) {
    const int j = c / (D / 8);
    const int col = (c % (D / 8)) * 8;
    const int jc = x * G + j;
    *reinterpret_cast<uint4*>(xk + j * D + col) =
        *reinterpret_cast<const uint4*>(combined_row(q, p, jc) + col);
    *reinterpret_cast<uint4*>(xv + j * D + col) =
        *reinterpret_cast<const uint4*>(combined_row_v(q, p, jc) + col);
  }
  __syncthreads();

  uint8_t* blk = q.g.blocks +
                 (static_cast<size_t>(p) * q.g.NB + q.first_block + x) * q.g.block_bytes;
  __half2* kmeta = reinterpret_cast<__half2*>(blk + q.g.off_km);
  __half2* vmeta = reinterpret_cast<__half2*>(blk + q.g.off_vm);

  // 2. statistics: D groups for K and D for V in every block, whatever the axis
  const int ng = D / G;  // channel groups per token (token axis)
  for (int e = tid; e < 2 * D; e += blockDim.x) {
    const bool isv = e >= D;
    const int ee = isv ? e - D : e;
    const int axis = isv ? q.g.av : q.g.ak;
    const int bits = isv ? q.g.bv : q.g.bk;
    const __half* base = isv ? xv : xk;
    Stat st;
    if (axis == 0) {  // channel ee over G tokens
      st = group_stat(base + ee, D, G, bits, (isv ? vmeta : kmeta) + ee);
    } else {          // token ee / ng, channels [(ee % ng) * G, +G)
      st = group_stat(base + (ee / ng) * D + (ee % ng) * G, 1, G, bits,
                      (isv ? vmeta : kmeta) + ee);
    }
    (isv ? sv : sk)[ee] = st;
  }
  __syncthreads();

  // 3a. K codes: token-major rows of D*bk/32 words
  {
    const int bits = q.g.bk;
    const int per = 32 / bits;
    const int kw = D * bits / 32;
    uint32_t* kc = reinterpret_cast<uint32_t*>(blk);
    for (int w = tid; w < G * kw; w += blockDim.x) {
      const int j = w / kw;
      const int d0 = (w % kw) * per;
      uint32_t word = 0;
      for (int e = 0; e < per; ++e) {
        const int d = d0 + e;
        const Stat st = sk[q.g.ak == 0 ? d : j * ng + d / G];
        word |= code_of(__half2float(xk[j * D + d]), st, bits) << (e * bits);
      }
      kc[w] = word;
    }
  }
  // 3b. V codes: 32-token chunks, channel-major, bv words per channel
  {
    const int bits = q.g.bv;
    const int per = 32 / bits;
    uint32_t* vc = reinterpret_cast<uint32_t*>(blk + q.g.off_vc);
    const int words = (G / 32) * D * bits;
    for (int w = tid; w < words; w += blockDim.x) {
      const int c = w / (D * bits);
      const int rem = w % (D * bits);
      const int d = rem / bits;
      const int j0 = c * 32 + (rem % bits) * per;
      uint32_t word = 0;
      for (int e = 0; e < per; ++e) {
        const int j = j0 + e;
        const Stat st = sv[q.g.av == 0 ? d : j * ng + d / G];
        word |= code_of(__half2float(xv[j * D + d]), st, bits) << (e * bits);
      }
      vc[w] = word;
    }
  }
}

__global__ void __launch_bounds__(kQuantThreads) dequantize_kernel(const DequantParams q) {
  const int i = blockIdx.x;
  const int p = blockIdx.y;
  const int D = q.g.D, G = q.g.G;
  const int ng = D / G;
  const uint8_t* blk =
      q.g.blocks + (static_cast<size_t>(p) * q.g.NB + i) * q.g.block_bytes;
  const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk);
  const __half2* km = reinterpret_cast<const __half2*>(blk + q.g.off_km);
  const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + q.g.off_vc);
  const __half2* vm = reinterpret_cast<const __half2*>(blk + q.g.off_vm);
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int j = e / D, d = e % D;
    const size_t o = (static_cast<size_t>(p) * q.T_q + static_cast<size_t>(i) * G + j) * D + d;
    {
      const int bits = q.g.bk, per = 32 / bits;
      const uint32_t word = kc[j * (D * bits / 32) + d / per];
      const uint32_t c = (word >> ((d % per) * bits)) & ((1u << bits) - 1u);
      const float2 sz = __half22float2(km[q.g.ak == 0 ? d : j * ng + d / G]);
      q.kout[o] = fmaf(static_cast<float>(c), sz.x, sz.y);
    }
    {
      const int bits = q.g.bv, per = 32 / bits;
      const int ch = j / 32, jj = j % 32;
      const uint32_t word = vc[(ch * D + d) * bits + jj / per];
      const uint32_t c = (word >> ((jj % per) * bits)) & ((1u << bits) - 1u);
      const float2 sz = __half22float2(vm[q.g.av == 0 ? d : j * ng + d / G]);
      q.vout[o] = fmaf(static_cast<float>(c), sz.x, sz.y);
    }
  }
}

size_t quantize_smem_bytes(int D, int G) {
  return static_cast<size_t>(2) * G * D * sizeof(__half) + 2 * D * sizeof(Stat);
}

// Opts the quantize kernel into the shared memory of the largest block
// (G = D = 128); called once per cache creation, with its device current.
cudaError_t prepare_quantize() {
  return cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(quantize_smem_bytes(128, 128)));
}

cudaError_t launch_quantize(const QuantParams& q, cudaStream_t stream) {
  const size_t smem = quantize_smem_bytes(q.g.D, q.g.G);
  dim3 grid(q.nflush + 1, q.g.P);
  quantize_kernel<<<grid, kQuantThreads, smem, stream>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const DequantParams& q, cudaStream_t stream) {
  dim3 grid(q.T_q / q.g.G, q.g.P);
  dequantize_kernel<<<grid, kQuantThreads, 0, stream>>>(q);
  return cudaGetLastError();
}

}  // namespace kvq
