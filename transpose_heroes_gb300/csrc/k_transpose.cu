// Transpose / layout-change hero kernels ("XLA:GPU Emitters", section "Transpose emitter": coalesced
// reads into a shared-memory tile, a barrier, coalesced writes out of it), and the element gathers.
//
//  tile_tma_kernel      -- the same for 4-byte elements when every stride allows 16-byte accesses:
//                          64 x 64 tiles by 2-D..5-D tensor copies into a ring of shared-memory
//                          stages, the prologue in place, 4 x 4 register transposes, 16-byte stores.
//  tile_transpose_kernel -- any physical permutation whose input-minor and output-minor axes
//                          differ: a 32 x 32 tile over those two axes, other axes batched.
//  gather_kernel        -- everything else: one thread per output element (also the quantized
//                          relayouts the tile kernel does not take, and broadcast_in_dim).
//  reshape_kernel       -- reshape with layouts: lexicographic position -> physical offsets.
#include <type_traits>

#include "async_copy.cuh"
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

// ---------------------------------------------------------------------------------------------
// Tensor-copy tile transpose (4-byte elements). Tile = 64 values of the input-minor axis a (one 256-byte
// row) x 64 of the output-minor axis b, at fixed batch coordinates; the tensor map's box is one tile,
// so a single copy fetches the 64 strided rows (elements outside the array read as 0 and are never
// stored). Thread t owns the 4 x 4 block (bi, bj) = (t / 16, t % 16): it reads b-rows 4bi.. (a values
// 4bj..) as 16-byte reads, applies the prologue, and after __syncwarp writes them back in place, 16-byte
// chunk c of row r at chunk c ^ ((r / 4) % 8) (its chunk lies in its own rows, read only by its half
// warp). After the block barrier it reads the block (bj, bi), transposes it in registers, applies the
// epilogue and stores output rows a = 4bi.. at b = 4bj.. with 16-byte stores. The last warp done with
// a stage refills it with the block's item j + NS (one barrier per item).
// ---------------------------------------------------------------------------------------------
constexpr int kTM = 64;
constexpr int kTmaTileStages = 4;
constexpr int kTileWarps = 8;

struct TileItem {
  int a0, b0;         // first a and b of the tile
  long long obase;    // output offset of the tile's batch coordinates
};

struct TileTmaShared {
  TileItem item[kTmaTileStages];
  int done[kTmaTileStages];
  uint64_t full[kTmaTileStages];
};

static size_t tile_tma_smem_bytes() {
  return 128 + (size_t)kTmaTileStages * kTM * kTM * 4 + sizeof(TileTmaShared);
}

// exp / log / tanh of four values through one out-of-line call (chains interpreted at run time)
static __device__ __noinline__ float4 chain_unary4(int op, float4 v, bool r16, int dt, const float4* lc,
                                                   const float2* le) {
  if (op == OP_EXP) return make_float4(chain_exp(v.x, r16, dt), chain_exp(v.y, r16, dt), chain_exp(v.z, r16, dt),
                                       chain_exp(v.w, r16, dt));
  if (op == OP_LOG)
    return make_float4(chain_log(v.x, r16, dt, lc, le), chain_log(v.y, r16, dt, lc, le),
                       chain_log(v.z, r16, dt, lc, le), chain_log(v.w, r16, dt, lc, le));
  return make_float4(chain_tanh(v.x, r16, dt), chain_tanh(v.y, r16, dt), chain_tanh(v.z, r16, dt),
                     chain_tanh(v.w, r16, dt));
}

// A chain (no broadcast operand) applied to four f32 values: one dispatch per op for all four.
__device__ __forceinline__ float4 apply_chain4(const Chain& c, float4 v, const LogTab& lt) {
  const float4 x = v;
  for (int k = 0; k < c.n; ++k) {
    const int op = c.op[k];
    const float imm = c.imm[k];
    switch (op) {
      case OP_EXP:
      case OP_LOG:
      case OP_TANH: v = chain_unary4(op, v, false, F32, lt.c, lt.e); break;
      case OP_ABS: v = make_float4(fabsf(v.x), fabsf(v.y), fabsf(v.z), fabsf(v.w)); break;
      case OP_NEG: v = make_float4(-v.x, -v.y, -v.z, -v.w); break;
      case OP_ADD_CONST:
        v = make_float4(__fadd_rn(v.x, imm), __fadd_rn(v.y, imm), __fadd_rn(v.z, imm), __fadd_rn(v.w, imm));
        break;
      case OP_MUL_CONST:
        v = make_float4(__fmul_rn(v.x, imm), __fmul_rn(v.y, imm), __fmul_rn(v.z, imm), __fmul_rn(v.w, imm));
        break;
      case OP_ADD_IN: v = make_float4(__fadd_rn(v.x, x.x), __fadd_rn(v.y, x.y), __fadd_rn(v.z, x.z), __fadd_rn(v.w, x.w)); break;
      case OP_MUL_IN: v = make_float4(__fmul_rn(v.x, x.x), __fmul_rn(v.y, x.y), __fmul_rn(v.z, x.z), __fmul_rn(v.w, x.w)); break;
      default: break;
    }
  }
  return v;
}

__device__ __forceinline__ float comp4(const float4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// PK: 0 -- no chains; 1 -- chains interpreted at run time; 2 -- the prologue is exactly exp (evaluated
// inline, its rare second and third passes out of line), the epilogue interpreted at run time.
// TK_EXP: the prologue is exactly exp (evaluated inline); TK_EXP_ABS: that, and the epilogue exactly abs
enum TileChains : int { TK_NONE = 0, TK_RT = 1, TK_EXP = 2, TK_EXP_ABS = 3 };
template <int PK>
__global__ void __launch_bounds__(256, 3)
    tile_tma_kernel(const __grid_constant__ CUtensorMap tmap, TilePlan p, int64_t nta, int64_t ntb, int64_t n_items) {
  constexpr bool CHAINS = PK != TK_NONE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  float* stage = reinterpret_cast<float*>(base);  // [stages][64 b-rows][64 a]
  TileTmaShared& ts = *reinterpret_cast<TileTmaShared*>(stage + kTmaTileStages * kTM * kTM);
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t na = p.size[p.ax_a], nb = p.size[p.ax_b];
  // copies item `it` (walk position j) into stage j % stages; records where its output goes
  auto issue = [&](int64_t it, int64_t j) {
    const int st = (int)(j % kTmaTileStages);
    int64_t rem = it;
    const int64_t ta = rem % nta;
    rem /= nta;
    const int64_t tb = rem % ntb;
    rem /= ntb;
    int32_t c[5] = {(int32_t)(ta * kTM), (int32_t)(tb * kTM), 0, 0, 0};
    int64_t obase = 0;
    for (int q = p.nbatch_axes - 1; q >= 0; --q) {  // batch coordinates, minor batch axis fastest
      const int ax = p.batch_axis[q];
      const int64_t i = rem % p.size[ax];
      rem /= p.size[ax];
      c[2 + q] = (int32_t)i;
      obase += i * p.out_stride[ax];
    }
    ts.item[st].a0 = c[0];
    ts.item[st].b0 = c[1];
    ts.item[st].obase = obase;
    const uint32_t bar = smem_addr(&ts.full[st]);
    mbar_arrive_expect_tx(bar, kTM * kTM * 4);
    float* dst = stage + st * kTM * kTM;
    const uint64_t map = reinterpret_cast<uint64_t>(&tmap);
    switch (2 + p.nbatch_axes) {
      case 2:
        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                     ::"r"(smem_addr(dst)), "l"(map), "r"(c[0]), "r"(c[1]), "r"(bar) : "memory");
        break;
      case 3:
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
                     ::"r"(smem_addr(dst)), "l"(map), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(bar) : "memory");
        break;
      case 4:
        asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
                     ::"r"(smem_addr(dst)), "l"(map), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(bar) : "memory");
        break;
      default:
        asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
                     ::"r"(smem_addr(dst)), "l"(map), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(bar) : "memory");
        break;
    }
  };
  if (tid == 0) {
    prefetch_tensor_map(&tmap);
    for (int st = 0; st < kTmaTileStages; ++st) {
      mbar_init(smem_addr(&ts.full[st]), 1);
      ts.done[st] = 0;
    }
    fence_mbar_init();
    for (int64_t j = 0; j < kTmaTileStages; ++j) {
      const int64_t it = blockIdx.x + j * gridDim.x;
      if (it < n_items) issue(it, j);
    }
  }
  __syncthreads();
  const LogTab lt = global_log_tables();
  float* out = reinterpret_cast<float*>(p.out);
  const int64_t soa = p.out_stride[p.ax_a];
  const int bi = tid >> 4, bj = tid & 15;
  const int own = 4 * bi * kTM + ((bj ^ (bi & 7)) << 2);  // b-row 4*bi, chunk bj (swizzled)
  const int oth = 4 * bj * kTM + ((bi ^ (bj & 7)) << 2);  // b-row 4*bj, chunk bi (swizzled)
  const int raw = 4 * bi * kTM + 4 * bj;                  // b-row 4*bi, a values 4*bj..
  int64_t j = 0;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
    const int st = (int)(j % kTmaTileStages);
    const bool arrived = mbar_wait(smem_addr(&ts.full[st]), (uint32_t)((j / kTmaTileStages) & 1));
    const TileItem ti = ts.item[st];
    float* tile = stage + st * kTM * kTM;
    // one b-row at a time: a thread's swizzled chunk of row r lies in row r, which only its own half
    // warp reads, so a warp sync per row orders the in-place rewrite; the loop keeps the code small
    // (fully unrolled, sixteen inline exps overflowed the instruction cache: 734 against 634 us)
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      float4 v = *reinterpret_cast<const float4*>(tile + raw + k * kTM);
      if (PK == TK_EXP || PK == TK_EXP_ABS) {  // two packed first passes; open ones (~1 in 2000) out of line
        float4 y;
        bool ok[4];
        cr_expf_first2(v.x, v.y, y.x, y.y, ok[0], ok[1]);
        cr_expf_first2(v.z, v.w, y.z, y.w, ok[2], ok[3]);
        if (!ok[0]) y.x = cr_expf_rest(v.x);
        if (!ok[1]) y.y = cr_expf_rest(v.y);
        if (!ok[2]) y.z = cr_expf_rest(v.z);
        if (!ok[3]) y.w = cr_expf_rest(v.w);
        v = y;
      }
      else if (CHAINS && p.pro.n) v = apply_chain4(p.pro, v, lt);
      __syncwarp();
      *reinterpret_cast<float4*>(tile + own + k * kTM) = v;
    }
    if (__syncthreads_or(arrived ? 0 : 1)) {
      if (tid == 0) {
        record_fault(kFaultCopyTimeout);
        for (int64_t q = j; q < j + kTmaTileStages && blockIdx.x + q * gridDim.x < n_items; ++q)
          mbar_wait(smem_addr(&ts.full[q % kTmaTileStages]), (uint32_t)((q / kTmaTileStages) & 1));
      }
      return;
    }
    float4 b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) b[k] = *reinterpret_cast<const float4*>(tile + oth + k * kTM);
    // the stage's values are in registers now: the last warp out refills it
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&ts.done[st], 1) == kTileWarps - 1) {
        ts.done[st] = 0;
        const int64_t nxt = item + (int64_t)kTmaTileStages * gridDim.x;
        if (nxt < n_items) {
          fence_proxy_async();
          issue(nxt, j + kTmaTileStages);
        }
      }
    }
    // output row a = a0 + 4bi + k holds b = b0 + 4bj + q: element (b-row 4bj + q, a 4bi + k) of the tile
    const int64_t b_first = ti.b0 + 4 * bj;
    if (b_first < nb) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t a = ti.a0 + 4 * bi + k;
        if (a >= na) break;
        float4 o = make_float4(comp4(b[0], k), comp4(b[1], k), comp4(b[2], k), comp4(b[3], k));
        if (PK == TK_EXP_ABS) o = make_float4(fabsf(o.x), fabsf(o.y), fabsf(o.z), fabsf(o.w));
        else if (CHAINS && p.epi.n) o = apply_chain4(p.epi, o, lt);
        *reinterpret_cast<float4*>(out + ti.obase + a * soa + b_first) = o;
      }
    }
  }
}

// A tensor map over the canonical input: dims (a, b, batch axes...), strides in bytes, 64 x 64 boxes.
static bool make_tile_tensor_map(const TilePlan& p, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const int rank = 2 + p.nbatch_axes;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5];
  dims[0] = (cuuint64_t)p.size[p.ax_a];
  dims[1] = (cuuint64_t)p.size[p.ax_b];
  strides[0] = (cuuint64_t)p.in_stride[p.ax_b] * 4;
  for (int q = 0; q < p.nbatch_axes; ++q) {
    dims[2 + q] = (cuuint64_t)p.size[p.batch_axis[q]];
    strides[1 + q] = (cuuint64_t)p.in_stride[p.batch_axis[q]] * 4;
  }
  for (int d = 0; d < rank; ++d) {
    box[d] = d < 2 ? kTM : 1;
    es[d] = 1;
  }
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void*>(p.in), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-copy tile path applies: 4-byte elements (f32 chains), at most three batch axes, every input
// stride but a's and every output stride but b's a multiple of 4 elements, dims within int32, aligned
// buffers, and nb a multiple of 4 (so a 16-byte store never straddles the end of b).
static bool tile_tma_ok(const TilePlan& p) {
  if (dt_bytes(p.dt) != 4 || p.nbatch_axes > 3) return false;
  if ((uintptr_t)p.in % 16 != 0 || (uintptr_t)p.out % 16 != 0) return false;
  if (p.size[p.ax_b] % 4 != 0) return false;
  if (p.in_stride[p.ax_a] != 1 || p.out_stride[p.ax_b] != 1) return false;
  for (int j = 0; j < p.k; ++j) {
    if (p.size[j] > 0x7FFFFFFF) return false;
    if (j != p.ax_a && p.in_stride[j] % 4 != 0) return false;
    if (j != p.ax_b && p.out_stride[j] % 4 != 0) return false;
  }
  return !chain_has_bcast_dev(p.pro) && !chain_has_bcast_dev(p.epi);
}

cudaError_t launch_tile_transpose(const TilePlan& p, cudaStream_t s) {
  const int64_t nta = (p.size[p.ax_a] + kTT - 1) / kTT;
  const int64_t ntb = (p.size[p.ax_b] + kTT - 1) / kTT;
  const int64_t blocks = nta * ntb * p.n_batch;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const bool chains = p.pro.n > 0 || p.epi.n > 0;
  CUtensorMap map;
  if (tile_tma_ok(p) && make_tile_tensor_map(p, &map)) {
    const int64_t nta64 = (p.size[p.ax_a] + kTM - 1) / kTM, ntb64 = (p.size[p.ax_b] + kTM - 1) / kTM;
    const int64_t items = nta64 * ntb64 * p.n_batch;
    const bool exp_pro = p.pro.n == 1 && p.pro.op[0] == OP_EXP;
    const bool abs_epi = p.epi.n == 1 && p.epi.op[0] == OP_ABS;
    auto kernel = !chains               ? tile_tma_kernel<TK_NONE>
                  : exp_pro && abs_epi ? tile_tma_kernel<TK_EXP_ABS>
                  : exp_pro            ? tile_tma_kernel<TK_EXP>
                                       : tile_tma_kernel<TK_RT>;
    const size_t smem = tile_tma_smem_bytes();
    const int nb = kernel_blocks_per_sm((const void*)kernel, 256, smem);
    int64_t grid = (int64_t)device_sm_count() * nb;
    if (grid > items) grid = items;
    kernel<<<(unsigned)grid, 256, smem, s>>>(map, p, nta64, ntb64, items);
    return cudaGetLastError();
  }
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
