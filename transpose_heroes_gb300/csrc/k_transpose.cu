// Transpose / layout-change hero kernels ("XLA:GPU Emitters", section "Transpose emitter": coalesced
// reads into a shared-memory tile, a barrier, coalesced writes out of it), and the element gathers.
//
//  tile_transpose_kernel -- any physical permutation whose input-minor and output-minor axes
//                          differ: a 32 x 32 tile over those two axes, other axes batched.
//  gather_kernel        -- everything else: one thread per output element (also the quantized
//                          relayouts the tile kernel does not take, and broadcast_in_dim).
//  reshape_kernel       -- reshape with layouts: lexicographic position -> physical offsets.
#include <type_traits>

#include "device_common.cuh"
#include "quant_common.cuh"

namespace hlo {

// ---------------------------------------------------------------------------------------------
// generic tiled transpose over canonical axes
// ---------------------------------------------------------------------------------------------
constexpr int kTT = 32;

template <typename T, bool CHAINS>
__global__ void __launch_bounds__(256) tile_transpose_kernel(TilePlan p, int64_t nta, int64_t ntb) {
  __shared__ T tile[kTT][kTT + 1];
  __shared__ float ftile[CHAINS ? kTT : 1][CHAINS ? kTT + 1 : 1];
  int64_t bid = blockIdx.x;
  const int64_t tA = bid % nta;
  bid /= nta;
  const int64_t tB = bid % ntb;
  const int64_t batch = bid / ntb;
  int64_t in_base = 0, out_base = 0, rem = batch;
  for (int j = p.nbatch_axes - 1; j >= 0; --j) {
    const int ax = p.batch_axis[j];
    const int64_t i = rem % p.size[ax];
    rem /= p.size[ax];
    in_base += i * p.in_stride[ax];
    out_base += i * p.out_stride[ax];
  }
  const int64_t a0 = tA * kTT, b0 = tB * kTT;
  const int64_t na = p.size[p.ax_a], nbb = p.size[p.ax_b];
  const int64_t sib = p.in_stride[p.ax_b], soa = p.out_stride[p.ax_a];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const T* in = reinterpret_cast<const T*>(p.in);
  T* out = reinterpret_cast<T*>(p.out);
  const LogTab lt = global_log_tables();
#pragma unroll
  for (int k = 0; k < kTT / 8; ++k) {
    const int r = ty + 8 * k;
    const int64_t a = a0 + tx, b = b0 + r;
    if (a < na && b < nbb) {
      if (CHAINS) {
        float v = load_as_f32(p.in, p.dt, in_base + b * sib + a);
        ftile[r][tx] = apply_chain_rt(p.pro, v, 0, lt);
      } else {
        tile[r][tx] = in[in_base + b * sib + a];
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kTT / 8; ++k) {
    const int r = ty + 8 * k;  // a within tile
    const int64_t a = a0 + r, b = b0 + tx;
    if (a < na && b < nbb) {
      if (CHAINS) {
        float v = apply_chain_rt(p.epi, ftile[tx][r], 0, lt);
        store_from_f32(p.out, p.dt, out_base + a * soa + b, round_to_dt(v, p.dt));
      } else {
        out[out_base + a * soa + b] = tile[tx][r];
      }
    }
  }
}

cudaError_t launch_tile_transpose(const TilePlan& p, cudaStream_t s) {
  const int64_t nta = (p.size[p.ax_a] + kTT - 1) / kTT;
  const int64_t ntb = (p.size[p.ax_b] + kTT - 1) / kTT;
  const int64_t blocks = nta * ntb * p.n_batch;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const bool chains = p.pro.n > 0 || p.epi.n > 0;
  if (chains) {
    tile_transpose_kernel<uint32_t, true><<<(unsigned)blocks, 256, 0, s>>>(p, nta, ntb);
  } else {
    switch (dt_bytes(p.dt)) {
      case 1: tile_transpose_kernel<uint8_t, false><<<(unsigned)blocks, 256, 0, s>>>(p, nta, ntb); break;
      case 2: tile_transpose_kernel<uint16_t, false><<<(unsigned)blocks, 256, 0, s>>>(p, nta, ntb); break;
      default: tile_transpose_kernel<uint32_t, false><<<(unsigned)blocks, 256, 0, s>>>(p, nta, ntb); break;
    }
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// general gather
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_kernel(GatherPlan p) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.n) return;
  const LogTab lt = global_log_tables();
  int64_t r[kMaxRank];
  int64_t rem = e;
  for (int j = p.rank - 1; j >= 0; --j) {
    const int64_t sz = p.out_size[j];
    r[p.out_logical[j]] = rem % sz;
    rem /= sz;
  }
  int64_t off = 0, self_off = 0, boff = 0, self_boff = 0;
  for (int k = 0; k < p.rank; ++k) {
    off += r[k] * p.in_stride_of_out[k];
    self_off += r[k] * p.self_stride_of_out[k];
    boff += r[k] * p.pro.bstride[p.perm[k]];
    self_boff += r[k] * p.pro.bstride[k];
  }
  if (p.kind == G_PLAIN) {
    if (p.pro.n == 0 && p.epi.n == 0 && !p.self_add) {
      const char* src = reinterpret_cast<const char*>(p.in) + off * p.elem_bytes;
      char* dst = reinterpret_cast<char*>(p.out) + e * p.elem_bytes;
      for (int b = 0; b < p.elem_bytes; ++b) dst[b] = src[b];
      return;
    }
    float v = apply_chain_rt(p.pro, load_as_f32(p.in, p.in_dt, off), boff, lt);
    if (p.self_add) {
      const float s = apply_chain_rt(p.pro, load_as_f32(p.in, p.in_dt, self_off), self_boff, lt);
      v = round_to_dt(__fadd_rn(s, v), p.pro.round16 ? p.in_dt : F32);
    }
    v = apply_chain_rt(p.epi, v, 0, lt);
    store_from_f32(p.out, p.out_dt, e, round_to_dt(v, p.out_dt));
    return;
  }
  // quantized: dequantize (input axis), float chain, quantize or f32 output
  const int code = (int)reinterpret_cast<const int8_t*>(p.in)[off];
  float sin = p.qin.scale;
  int zin = p.qin.zp;
  if (p.qin_axis_out >= 0) {
    const int64_t j = r[p.qin_axis_out];
    sin = p.qin.scales[j];
    zin = p.qin.zps[j];
  }
  float real = dequant(code, sin, zin);
  real = apply_chain_rt(p.pro, real, boff, lt);
  if (p.out_float) {
    reinterpret_cast<float*>(p.out)[e] = real;
    return;
  }
  float sout = p.qout.scale, inv = p.qout.inv_scale;
  int zout = p.qout.zp;
  if (p.qout_axis_out >= 0) {
    const int64_t j = r[p.qout_axis_out];
    sout = p.qout.scales[j];
    zout = p.qout.zps[j];
    inv = __frcp_rn(sout);
  }
  reinterpret_cast<int8_t*>(p.out)[e] = (int8_t)quant_code(real, sout, inv, zout, p.qout.smin, p.qout.smax);
}

// ---------------------------------------------------------------------------------------------
// reshape and the parameters of quantized data movement
// ---------------------------------------------------------------------------------------------
template <int EB>
__global__ void __launch_bounds__(256) reshape_kernel(ReshapePlan p) {
  using T = typename std::conditional<EB == 4, uint32_t, typename std::conditional<EB == 2, uint16_t, uint8_t>::type>::type;
  const T* in = reinterpret_cast<const T*>(p.in);
  T* out = reinterpret_cast<T*>(p.out);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.n; e += (int64_t)gridDim.x * blockDim.x)
    out[e] = in[map_index(p.lex_to_in, map_index(p.out_to_lex, e))];
}

cudaError_t launch_reshape(const ReshapePlan& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  int64_t blocks = (p.n + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (p.elem_bytes == 4) reshape_kernel<4><<<(unsigned)blocks, 256, 0, s>>>(p);
  else if (p.elem_bytes == 2) reshape_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(p);
  else reshape_kernel<1><<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

__global__ void quant_params_kernel(const float* src_s, const int32_t* src_z, float s0, int32_t z0, int single,
                                    float* dst_s, int32_t* dst_z, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = single ? 0 : i;
    dst_s[i] = src_s ? src_s[k] : s0;
    dst_z[i] = src_s ? src_z[k] : z0;
  }
}

cudaError_t launch_quant_params(const float* src_s, const int32_t* src_z, float s0, int32_t z0, int single, float* dst_s,
                                int32_t* dst_z, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  quant_params_kernel<<<(unsigned)blocks, 256, 0, s>>>(src_s, src_z, s0, z0, single, dst_s, dst_z, n);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherPlan& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const int64_t blocks = (p.n + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  gather_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hlo
