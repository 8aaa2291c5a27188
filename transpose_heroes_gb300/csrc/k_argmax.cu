// Variadic reduce with the max/argmax body ("XLA Operation Semantics", section "Variadic Reduce"):
// f(max, argmax, value, index) = (value, index) if value >= max else (max, argmax), from (I_V, I_K).
//
//  argmax_row_kernel -- the reduced walk is contiguous in memory: a block per output, threads take
//                       16-byte vectors in turn (four loads in flight, each folded into its own
//                       partial in increasing position), then the partials combine in the thread and
//                       the block (warp shuffles + shared memory).
//  argmax_gen_kernel -- anything else: a thread per output walks the reduced positions in order
//                       (adjacent threads read adjacent outputs' elements, so a reduced major
//                       dimension streams coalesced).
// Partials carry the walk position of the element they selected (-1: none, the init). Folding in
// increasing position with value >= max is f itself; two partials combine to the greater value, or on
// equal values to the later position: the element the sequential fold over both would keep. The
// index K is read once per output, at the final position.
#include "device_common.cuh"

namespace hlo {

struct Best {
  float v;
  long long pos;
};

__device__ __forceinline__ void fold(Best& b, float x, long long pos) {
  if (x >= b.v) {  // false for NaN: a NaN value is never selected
    b.v = x;
    b.pos = pos;
  }
}

__device__ __forceinline__ Best later_max(Best a, Best b) {
  return (b.v > a.v || (b.v == a.v && b.pos > a.pos)) ? b : a;
}

__device__ __forceinline__ void write_result(const ArgmaxPlan& p, int64_t o, Best b) {
  store_from_f32(p.out, p.dt, map_index(p.okept, o), b.v);
  int32_t idx = p.init_index;
  if (b.pos >= 0) idx = p.k ? p.k[map_index(p.kkept, o) + map_index(p.kred, b.pos)] : (int32_t)b.pos;
  p.out_idx[map_index(p.ikept, o)] = idx;
}

template <int DT>
__device__ __forceinline__ void fold_vec(Best& b, uint4 w, long long pos0) {
  if (DT == F32) {
    fold(b, __uint_as_float(w.x), pos0);
    fold(b, __uint_as_float(w.y), pos0 + 1);
    fold(b, __uint_as_float(w.z), pos0 + 2);
    fold(b, __uint_as_float(w.w), pos0 + 3);
  } else {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = DT == BF16 ? __uint_as_float(ws[j] << 16) : f16_bits_to_f32((uint16_t)(ws[j] & 0xFFFFu));
      const float hi = DT == BF16 ? __uint_as_float(ws[j] & 0xFFFF0000u) : f16_bits_to_f32((uint16_t)(ws[j] >> 16));
      fold(b, lo, pos0 + 2 * j);
      fold(b, hi, pos0 + 2 * j + 1);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(256) argmax_row_kernel(ArgmaxPlan p, int vec) {
  __shared__ float sv[8];
  __shared__ long long sp[8];
  constexpr int E = DT == F32 ? 4 : 8;  // elements per 16-byte vector
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t o = blockIdx.x; o < p.n_out; o += gridDim.x) {
    const int64_t base = map_index(p.vkept, o);
    Best b{p.init_value, -1};
    if (vec) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.v) + base * (DT == F32 ? 4 : 2));
      const int64_t nv = p.n_red / E, bd = blockDim.x;
      Best b4[4] = {b, b, b, b};
      int64_t q = threadIdx.x;
      for (; q + 3 * bd < nv; q += 4 * bd) {
        const uint4 w0 = __ldg(src + q), w1 = __ldg(src + q + bd), w2 = __ldg(src + q + 2 * bd), w3 = __ldg(src + q + 3 * bd);
        fold_vec<DT>(b4[0], w0, q * E);
        fold_vec<DT>(b4[1], w1, (q + bd) * E);
        fold_vec<DT>(b4[2], w2, (q + 2 * bd) * E);
        fold_vec<DT>(b4[3], w3, (q + 3 * bd) * E);
      }
      for (; q < nv; q += bd) fold_vec<DT>(b4[0], __ldg(src + q), q * E);  // later positions than b4[0] holds
      b = later_max(later_max(b4[0], b4[1]), later_max(b4[2], b4[3]));
    } else {
      for (int64_t t = threadIdx.x; t < p.n_red; t += blockDim.x) fold(b, load_as_f32(p.v, DT, base + t), t);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      Best c;
      c.v = __shfl_xor_sync(0xffffffffu, b.v, off);
      c.pos = __shfl_xor_sync(0xffffffffu, b.pos, off);
      b = later_max(b, c);
    }
    if (lane == 0) {
      sv[warp] = b.v;
      sp[warp] = b.pos;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      Best r{sv[0], sp[0]};
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = later_max(r, Best{sv[w], sp[w]});
      write_result(p, o, r);
    }
    __syncthreads();  // sv/sp are reused by the next output
  }
}

template <int DT>
__global__ void __launch_bounds__(256) argmax_gen_kernel(ArgmaxPlan p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < p.n_out; o += stride) {
    const int64_t base = map_index(p.vkept, o);
    Best b{p.init_value, -1};
    if (p.vred.identity || p.vred.n == 1) {
      const int64_t rs = p.vred.identity ? 1 : p.vred.stride[0];
      for (int64_t t = 0; t < p.n_red; ++t) fold(b, load_as_f32(p.v, DT, base + t * rs), t);
    } else {
      for (int64_t t = 0; t < p.n_red; ++t) fold(b, load_as_f32(p.v, DT, base + map_index(p.vred, t)), t);
    }
    write_result(p, o, b);
  }
}

cudaError_t launch_argmax(const ArgmaxPlan& p, cudaStream_t s) {
  if (p.n_out == 0) return cudaSuccess;
  const int eb = dt_bytes(p.dt);
  if (p.vred.identity && p.n_red >= 256) {
    // 16-byte vectors when every output's walk starts on a 16-byte boundary and is whole vectors long
    const int E = 16 / eb;
    bool vec = ((uintptr_t)p.v % 16 == 0) && (p.n_red % E == 0);
    if (vec && p.n_out > 1) {
      // bases differ by the kept strides; all must be multiples of E elements
      for (int j = 0; j < p.vkept.n; ++j) vec = vec && (p.vkept.stride[j] % E == 0);
      if (p.vkept.identity) vec = false;  // a stride of 1 between outputs is never a whole vector
    }
    // one wave of resident blocks, every block with the same number of outputs (give or take one)
    const void* kernel = p.dt == F32 ? (const void*)argmax_row_kernel<F32>
                         : p.dt == BF16 ? (const void*)argmax_row_kernel<BF16> : (const void*)argmax_row_kernel<F16>;
    const int64_t cap = (int64_t)device_sm_count() * kernel_blocks_per_sm(kernel, 256, 0);
    const int64_t per = (p.n_out + cap - 1) / cap;
    const int64_t grid = (p.n_out + per - 1) / per;
    if (p.dt == F32) argmax_row_kernel<F32><<<(unsigned)grid, 256, 0, s>>>(p, vec ? 1 : 0);
    else if (p.dt == BF16) argmax_row_kernel<BF16><<<(unsigned)grid, 256, 0, s>>>(p, vec ? 1 : 0);
    else argmax_row_kernel<F16><<<(unsigned)grid, 256, 0, s>>>(p, vec ? 1 : 0);
    return cudaGetLastError();
  }
  int64_t grid = (p.n_out + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (grid > cap) grid = cap;
  if (p.dt == F32) argmax_gen_kernel<F32><<<(unsigned)grid, 256, 0, s>>>(p);
  else if (p.dt == BF16) argmax_gen_kernel<BF16><<<(unsigned)grid, 256, 0, s>>>(p);
  else argmax_gen_kernel<F16><<<(unsigned)grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hlo
