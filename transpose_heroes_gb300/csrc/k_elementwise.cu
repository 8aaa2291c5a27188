// Elementwise kernel for fusions whose transpose is the identity on memory (same physical order in and
// out): the loop emitter of "XLA:GPU Emitters" (section "Loop emitter": a linear walk over the output
// so that writes are coalesced, with vectorized loads and stores, section "Vectorization").
#include "device_common.cuh"

namespace hlo {

struct EwPlan {
  const void* in;
  void* out;
  int64_t n;
  int dt;
  Chain pro, epi;
};

__device__ __forceinline__ float ew_apply(const EwPlan& p, float v, const LogTab& lt) {
  v = apply_chain_rt<false>(p.pro, v, 0, lt);
  return apply_chain_rt<false>(p.epi, v, 0, lt);
}

// Two elements of log through the first pass, the rest of the correctly rounded log where it
// leaves the rounding open (same result as cr_logf).
__device__ __forceinline__ void log2x(float& a, float& b, const float* l1i, const float* l1h, const float* l1l,
                                      const LogTab& lt) {
  float ya, yb;
  bool oa, ob;
  cr_logf_first2(a, b, l1i, l1h, l1l, ya, yb, oa, ob);
  a = oa ? ya : cr_logf(a, lt.c, lt.e);
  b = ob ? yb : cr_logf(b, lt.c, lt.e);
}

template <bool VEC>
__global__ void __launch_bounds__(256) elementwise_f32_kernel(EwPlan p) {
  __shared__ float4 s_lc[HLO_LOG_NC];
  __shared__ float2 s_le[HLO_LOG_NE];
  __shared__ float s_l1[3][32];
  load_log_tables(s_lc, s_le);
  load_log1_tables(s_l1[0], s_l1[1], s_l1[2]);
  __syncthreads();
  const LogTab lt = {s_lc, s_le};
  const bool pure_log = p.pro.n == 1 && p.pro.op[0] == OP_LOG && p.epi.n == 0;
  const float* in = reinterpret_cast<const float*>(p.in);
  float* out = reinterpret_cast<float*>(p.out);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (VEC) {
    const int64_t nv = p.n / 4;
    for (int64_t v = tid; v < nv; v += stride) {
      float4 x = __ldg(reinterpret_cast<const float4*>(in) + v);
      if (pure_log) {
        log2x(x.x, x.y, s_l1[0], s_l1[1], s_l1[2], lt);
        log2x(x.z, x.w, s_l1[0], s_l1[1], s_l1[2], lt);
      } else {
        x.x = ew_apply(p, x.x, lt);
        x.y = ew_apply(p, x.y, lt);
        x.z = ew_apply(p, x.z, lt);
        x.w = ew_apply(p, x.w, lt);
      }
      reinterpret_cast<float4*>(out)[v] = x;
    }
    done = nv * 4;
  }
  for (int64_t e = done + tid; e < p.n; e += stride) out[e] = ew_apply(p, in[e], lt);
}

__global__ void __launch_bounds__(256) elementwise_any_kernel(EwPlan p) {
  const LogTab lt = global_log_tables();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.n; e += stride) {
    float v = ew_apply(p, load_as_f32(p.in, p.dt, e), lt);
    store_from_f32(p.out, p.dt, e, round_to_dt(v, p.dt));
  }
}

// Pure data movement with identical memory order: raw bytes, 16 at a time where aligned.
__global__ void __launch_bounds__(256) copy_bytes_kernel(const uint8_t* in, uint8_t* out, int64_t nbytes, bool vec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t nv = nbytes / 16;
    for (int64_t v = tid; v < nv; v += stride)
      reinterpret_cast<uint4*>(out)[v] = __ldg(reinterpret_cast<const uint4*>(in) + v);
    done = nv * 16;
  }
  for (int64_t b = done + tid; b < nbytes; b += stride) out[b] = in[b];
}

cudaError_t launch_copy(const void* in, void* out, int64_t nbytes, cudaStream_t s) {
  if (nbytes == 0) return cudaSuccess;
  int64_t blocks = (nbytes + 4095) / 4096;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const bool vec = ((uintptr_t)in % 16 == 0) && ((uintptr_t)out % 16 == 0);
  copy_bytes_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const uint8_t*>(in),
                                                      reinterpret_cast<uint8_t*>(out), nbytes, vec);
  return cudaGetLastError();
}

cudaError_t launch_elementwise(const void* in, void* out, int64_t n, int dt, const Chain& pro, const Chain& epi,
                               cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  EwPlan p{in, out, n, dt, pro, epi};
  int64_t blocks = (n + 1023) / 1024;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dt == F32) {
    const bool vec = ((uintptr_t)in % 16 == 0) && ((uintptr_t)out % 16 == 0);
    if (vec) elementwise_f32_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(p);
    else elementwise_f32_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(p);
  } else {
    elementwise_any_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace hlo
