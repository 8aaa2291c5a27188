// Reduce-hero kernels ("StableHLO Specification", section "reduce"; "XLA:GPU Emitters": the reduction
// emitter reduces with warp shuffles and shared memory).
//
//  row_reduce_kernel  -- reduced dimensions are the minor-most physical ones: the input is [K, R] with
//                        rows contiguous. Persistent blocks walk rows; every thread streams 16-byte
//                        vectors of the row, applies the prologue in registers and accumulates in f32;
//                        the block combines through warp shuffles and shared memory.
//  col_reduce_kernel  -- kept dimensions on both sides: the input is [A, R, B] with B contiguous.
//                        A thread owns one 16-byte column vector; the 8 warps of a block split the rows
//                        of a slab; a thread-block cluster of kColCluster blocks splits R into slabs and
//                        block rank 0 combines the slab partials read from the others' shared memory
//                        (distributed shared memory), so one launch produces the output, no workspace.
//  gen_reduce_kernel  -- any other pattern: one thread per output element.
#include <cooperative_groups.h>

#include "async_copy.cuh"
#include "device_common.cuh"

namespace cg = cooperative_groups;

namespace hlo {

// Compiled prologue chains of the row kernel.
enum RowChain : int { RC_NONE = 0, RC_EXP = 1, RC_EXP_BCAST_BF16 = 2, RC_RT = 3 };

constexpr int kRowThreads = 512;
constexpr int kRowUnroll = 4;

template <int KIND>
__device__ __forceinline__ float block_reduce(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = combine<KIND>(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  if (warp == 0) {
    v = lane < nw ? red[lane] : identity<KIND>();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = combine<KIND>(v, __shfl_xor_sync(0xffffffffu, v, o));
  }
  __syncthreads();
  return v;  // valid in thread 0
}

__device__ __forceinline__ void store_result(void* out, int dt, int64_t off, float v) {
  store_from_f32(out, dt, off, v);
}

// ---- element kernels of the row reduce --------------------------------------------------------
// Processes one 16-byte vector: f32 x4 or 16-bit x8.
template <int IN_DT, int CH, int KIND>
__device__ __forceinline__ float row_vec(uint4 x, uint4 b, float acc, const Chain& ch, const LogTab& lt) {
  if (IN_DT == F32) {
    float v[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z), __uint_as_float(x.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t = v[i];
      if (CH == RC_EXP) t = KIND == RED_ADD ? fast_exp(t) : cr_expf(t);
      if (CH == RC_RT) t = apply_chain_rt(ch, t, 0, lt);
      acc = combine<KIND>(acc, t);
    }
    return acc;
  } else {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    float part = identity<KIND>();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      if (IN_DT == BF16) {
        lo = bf16_bits_to_f32(w[i] & 0xFFFFu);
        hi = __uint_as_float(w[i] & 0xFFFF0000u);
      } else {
        lo = f16_bits_to_f32((uint16_t)(w[i] & 0xFFFFu));
        hi = f16_bits_to_f32((uint16_t)(w[i] >> 16));
      }
      if (CH == RC_EXP_BCAST_BF16) {
        // bf16(exp(x)) then the bf16 add with the broadcast pair, rounded once (add.rn.bf16x2); a max
        // body keeps every term exact, so it takes the correctly rounded bf16 exp
        float elo, ehi;
        if (KIND == RED_ADD) {
          elo = fast_exp(lo);
          ehi = fast_exp(hi);
        } else {
          elo = chain_exp(lo, true, BF16);
          ehi = chain_exp(hi, true, BF16);
        }
        uint32_t e2, s2;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(e2) : "f"(ehi), "f"(elo));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(s2) : "r"(e2), "r"(bw[i]));
        lo = __uint_as_float(s2 << 16);
        hi = __uint_as_float(s2 & 0xFFFF0000u);
      } else {
        if (CH == RC_EXP) {
          if (KIND == RED_ADD) {
            lo = fast_exp(lo);
            hi = fast_exp(hi);
            if (ch.round16) {
              lo = round_to_dt(lo, IN_DT);
              hi = round_to_dt(hi, IN_DT);
            }
          } else {
            lo = chain_exp(lo, ch.round16, IN_DT);
            hi = chain_exp(hi, ch.round16, IN_DT);
          }
        }
        if (CH == RC_RT) {
          lo = apply_chain_rt(ch, lo, 0, lt);
          hi = apply_chain_rt(ch, hi, 0, lt);
        }
      }
      part = combine<KIND>(part, combine<KIND>(lo, hi));
    }
    return combine<KIND>(acc, part);
  }
}

// VEC = elements per 16-byte vector (4 for f32, 8 for 16-bit) or 1 for the scalar variant.
template <int IN_DT, int VEC, int CH, int KIND>
__global__ void __launch_bounds__(kRowThreads) row_reduce_kernel(RowReducePlan p) {
  __shared__ float red[32];
  __shared__ float4 s_lc[HLO_LOG_NC];
  __shared__ float2 s_le[HLO_LOG_NE];
  LogTab lt = global_log_tables();
  if (CH == RC_RT && chain_has_log(p.chain)) {
    load_log_tables(s_lc, s_le);
    __syncthreads();
    lt = {s_lc, s_le};
  }
  const int eb = IN_DT == F32 ? 4 : 2;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t n_items = p.rows * p.split;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    // item = (row, segment): elements [e0, e0 + len) of the row; e0 is a multiple of VEC
    const int64_t row = item / p.split, sg = item - row * p.split;
    const int64_t e0 = sg * p.seg;
    const int64_t len = min(p.seg, p.len - e0);
    const char* base = reinterpret_cast<const char*>(p.in) + (row * p.len + e0) * eb;
    float acc = identity<KIND>();
    int64_t tail_start = 0;
    if (VEC > 1) {
      const int64_t nvec = len / VEC;
      const uint4* xv = reinterpret_cast<const uint4*>(base);
      const uint4* bv = reinterpret_cast<const uint4*>(p.chain.bptr) + (CH == RC_EXP_BCAST_BF16 ? e0 / VEC : 0);
      int64_t v = tid;
      for (; v + (kRowUnroll - 1) * (int64_t)nt < nvec; v += kRowUnroll * (int64_t)nt) {
        uint4 x[kRowUnroll], b[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(x[u].x), "=r"(x[u].y), "=r"(x[u].z), "=r"(x[u].w)
                       : "l"(xv + v + u * nt));
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          if (CH == RC_EXP_BCAST_BF16) b[u] = __ldg(bv + v + u * nt);
          else b[u] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) acc = row_vec<IN_DT, CH, KIND>(x[u], b[u], acc, p.chain, lt);
      }
      for (; v < nvec; v += nt) {
        uint4 x = __ldg(xv + v);
        uint4 b = CH == RC_EXP_BCAST_BF16 ? __ldg(bv + v) : make_uint4(0, 0, 0, 0);
        acc = row_vec<IN_DT, CH, KIND>(x, b, acc, p.chain, lt);
      }
      tail_start = nvec * VEC;
    }
    // scalar elements (all of them for VEC == 1, the ragged tail otherwise)
    for (int64_t e = tail_start + tid; e < len; e += nt) {
      float t = load_as_f32(base, IN_DT, e);
      if (CH == RC_EXP) {
        if (KIND == RED_ADD) {
          t = fast_exp(t);
          if (p.chain.round16) t = round_to_dt(t, IN_DT);
        } else {
          t = chain_exp(t, p.chain.round16 && IN_DT != F32, IN_DT);
        }
      } else if (CH == RC_EXP_BCAST_BF16) {
        t = KIND == RED_ADD ? round_to_dt(fast_exp(t), BF16) : chain_exp(t, true, BF16);
        t = round_to_dt(__fadd_rn(t, load_as_f32(p.chain.bptr, BF16, e0 + e)), BF16);
      } else if (CH == RC_RT) {
        int64_t boff = p.bmode == BC_ROWVEC ? e0 + e : p.bmode == BC_PERROW ? map_index(p.bmap, row) : 0;
        t = apply_chain_rt(p.chain, t, boff, lt);
      }
      acc = combine<KIND>(acc, t);
    }
    acc = block_reduce<KIND>(acc, red);
    if (tid == 0) {
      if (p.split > 1) p.ws[item] = acc;  // the segment's partial, combined by row_split_combine_kernel
      else store_result(p.out, p.out_dt, map_index(p.omap, row), combine<KIND>(p.init, acc));
    }
  }
}

// Second pass of a split row reduce: one thread per row combines the row's segment partials in segment
// order (deterministic), then applies init once.
template <int KIND>
__global__ void row_split_combine_kernel(RowReducePlan p) {
  for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < p.rows;
       row += (int64_t)gridDim.x * blockDim.x) {
    const float* part = p.ws + row * p.split;
    float acc = part[0];
    for (int64_t sg = 1; sg < p.split; ++sg) acc = combine<KIND>(acc, part[sg]);
    store_result(p.out, p.out_dt, map_index(p.omap, row), combine<KIND>(p.init, acc));
  }
}

// ---- streaming row reduce (bulk asynchronous copies into a shared-memory ring) --------------------
// Rows are cut into chunks of up to kChunkBytes, kept in flight kStages at a time with 1-D bulk copies
// (cp.async.bulk, completion counted on one mbarrier per stage). Every warp consumes its share of a
// chunk from shared memory with 16-byte reads and then releases the stage on a shared counter; the
// warp whose release completes the count issues the copy of the chunk kStages ahead into that stage.
// At the end of a row each warp leaves its partial in a slot, and the warp that completes the slot
// combines the partials in warp order and stores the row. So no block-wide barrier stands in the
// stream: warps drift apart by at most kStages chunks. Bytes in flight do not depend on registers:
// up to kStages * kChunkBytes per block.
constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kChunkBytes = 16384;
constexpr int kStages = 3;
constexpr int kRowSlots = 8;  // > the rows kStages chunks can span, so a slot is free when reused
// Packed (float2) element work of the streaming row reduce for the add body: two independent
// f32 partial sums per thread, combined at the end of the row.
__device__ __forceinline__ float ex2_approx(float t) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

template <int IN_DT, int CH>
__device__ __forceinline__ float2 row_vec2_add(uint4 x, uint4 b, float2 acc) {
  const float2 l2e = make_float2(1.4426950408889634f, 1.4426950408889634f);
  if (IN_DT == F32) {
    float2 v0 = make_float2(__uint_as_float(x.x), __uint_as_float(x.y));
    float2 v1 = make_float2(__uint_as_float(x.z), __uint_as_float(x.w));
    if (CH == RC_EXP) {
      const float2 t0 = __fmul2_rn(v0, l2e), t1 = __fmul2_rn(v1, l2e);
      v0 = make_float2(ex2_approx(t0.x), ex2_approx(t0.y));
      v1 = make_float2(ex2_approx(t1.x), ex2_approx(t1.y));
    }
    return __fadd2_rn(__fadd2_rn(acc, v0), v1);
  } else {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 v = IN_DT == BF16 ? make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u))
                               : make_float2(f16_bits_to_f32((uint16_t)(w[i] & 0xFFFFu)),
                                             f16_bits_to_f32((uint16_t)(w[i] >> 16)));
      if (CH == RC_EXP_BCAST_BF16) {
        // bf16(exp(x)), then the bf16 add with the broadcast pair rounded once (add.rn.bf16x2), then
        // each bf16 sum added to its f32 partial in one instruction (the bf16 -> f32 widening is exact)
        const float2 t = __fmul2_rn(v, l2e);
        uint32_t e2, s2;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(e2) : "f"(ex2_approx(t.y)), "f"(ex2_approx(t.x)));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(s2) : "r"(e2), "r"(bw[i]));
        asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.bf16 %0, l, %0; add.rn.f32.bf16 %1, h, %1; }"
            : "+f"(acc.x), "+f"(acc.y)
            : "r"(s2));
        continue;
      }
      acc = __fadd2_rn(acc, v);
    }
    return acc;
  }
}

template <int IN_DT, int CH, int KIND, bool BREG>
__global__ void __launch_bounds__(kStreamThreads) row_stream_kernel(RowReducePlan p, int cpr) {
  extern __shared__ __align__(128) uint8_t ring[];  // kStages x kChunkBytes
  __shared__ __align__(8) uint64_t bar[kStages];
  __shared__ int stage_cnt[kStages];                 // warps done with the stage's current chunk
  __shared__ long long last_issued[kStages];         // last chunk copied into each stage
  __shared__ int row_cnt[kRowSlots];                 // warps done with the slot's row
  __shared__ float partial[kRowSlots][kStreamWarps];
  __shared__ volatile int abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int eb = IN_DT == F32 ? 4 : 2;
  const int64_t row_bytes = p.len * eb;
  const int64_t my_rows = p.rows > blockIdx.x ? (p.rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t n_chunks = my_rows * cpr;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&bar[s]), 1);
      stage_cnt[s] = 0;
      last_issued[s] = -1;
    }
    for (int r = 0; r < kRowSlots; ++r) row_cnt[r] = 0;
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  auto chunk_bytes = [&](int part) {
    const int64_t rem = row_bytes - (int64_t)part * kChunkBytes;
    return (uint32_t)(rem < kChunkBytes ? rem : kChunkBytes);
  };
  // copies chunk g (row `row`, part `part`) into stage g mod kStages
  auto issue = [&](int64_t g, int64_t row, int part) {
    const uint32_t bytes = chunk_bytes(part);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.in) + row * row_bytes + (int64_t)part * kChunkBytes;
    const int s = (int)(g % kStages);
    const uint32_t b = smem_addr(&bar[s]);
    last_issued[s] = g;
    fence_proxy_async();
    mbar_arrive_expect_tx(b, bytes);
    bulk_load(ring + s * kChunkBytes, src, bytes, b);
  };
  if (tid == 0) {
    int64_t row = blockIdx.x;
    int part = 0;
    for (int64_t g = 0; g < kStages && g < n_chunks; ++g) {
      issue(g, row, part);
      if (++part == cpr) {
        part = 0;
        row += gridDim.x;
      }
    }
  }
  const uint4* bv = reinterpret_cast<const uint4*>(p.chain.bptr);
  const LogTab lt = global_log_tables();
  // BREG: rows of at most two chunks; this thread's slice of the broadcast vector (the same for every
  // row) stays in registers: vectors tid + 256 k of each chunk.
  constexpr int kVecPerThread = kChunkBytes / 16 / kStreamThreads;
  uint4 breg[2][kVecPerThread];
  if (BREG) {
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const int64_t vi = (int64_t)part * (kChunkBytes / 16) + tid + k * kStreamThreads;
        breg[part][k] = (part < cpr && vi * 16 < row_bytes) ? __ldg(bv + vi) : make_uint4(0, 0, 0, 0);
      }
  }
  float acc = identity<KIND>();
  int cons_part = 0, cons_stage = 0, row_slot = 0;
  uint32_t cons_parity = 0;
  int64_t cons_row = blockIdx.x;
  // the chunk kStages ahead of the one being consumed: its row and part
  int64_t nxt_row = blockIdx.x + (int64_t)(kStages / cpr) * gridDim.x;
  int nxt_part = kStages % cpr;
  for (int64_t g = 0; g < n_chunks; ++g) {
    const int s = cons_stage;
    if (abort_flag) break;
    if (!mbar_wait(smem_addr(&bar[s]), cons_parity)) {
      abort_flag = 1;
      break;
    }
    const uint32_t bytes = chunk_bytes(cons_part);
    const int part = cons_part;
    const uint4* xv = reinterpret_cast<const uint4*>(ring + s * kChunkBytes);
    const int nv = (int)(bytes / 16);
    const int64_t vbase = part * (kChunkBytes / 16);  // vector index of the chunk within the row
    if (BREG) {
      float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const int v = tid + k * kStreamThreads;
        if (v < nv) acc2 = row_vec2_add<IN_DT, CH>(xv[v], part == 0 ? breg[0][k] : breg[1][k], acc2);
      }
      acc = __fadd_rn(acc, __fadd_rn(acc2.x, acc2.y));
    } else if (KIND == RED_ADD && CH != RC_RT && !(CH == RC_EXP && IN_DT != F32 && p.chain.round16)) {
      float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll 4
      for (int v = tid; v < nv; v += kStreamThreads) {
        const uint4 x = xv[v];
        const uint4 b = CH == RC_EXP_BCAST_BF16 ? __ldg(bv + vbase + v) : make_uint4(0, 0, 0, 0);
        acc2 = row_vec2_add<IN_DT, CH>(x, b, acc2);
      }
      acc = __fadd_rn(acc, __fadd_rn(acc2.x, acc2.y));
    } else {
#pragma unroll 4
      for (int v = tid; v < nv; v += kStreamThreads) {
        const uint4 x = xv[v];
        const uint4 b = CH == RC_EXP_BCAST_BF16 ? __ldg(bv + vbase + v) : make_uint4(0, 0, 0, 0);
        acc = row_vec<IN_DT, CH, KIND>(x, b, acc, p.chain, lt);
      }
    }
    __syncwarp();  // the warp's reads of stage s are done
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&stage_cnt[s], 1) == kStreamWarps - 1) {  // the last warp out refills the stage
        __threadfence_block();
        stage_cnt[s] = 0;
        if (g + kStages < n_chunks && !abort_flag) issue(g + kStages, nxt_row, nxt_part);
      }
    }
    if (part == cpr - 1) {  // end of the row: partial per warp; the warp completing the slot stores
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc = combine<KIND>(acc, __shfl_xor_sync(0xffffffffu, acc, o));
      if (lane == 0) {
        partial[row_slot][warp] = acc;
        __threadfence_block();
        if (atomicAdd(&row_cnt[row_slot], 1) == kStreamWarps - 1) {
          row_cnt[row_slot] = 0;
          __threadfence_block();
          float r = partial[row_slot][0];
#pragma unroll
          for (int w = 1; w < kStreamWarps; ++w) r = combine<KIND>(r, partial[row_slot][w]);
          store_result(p.out, p.out_dt, map_index(p.omap, cons_row), combine<KIND>(p.init, r));
        }
      }
      acc = identity<KIND>();
      cons_row += gridDim.x;
      row_slot = row_slot + 1 == kRowSlots ? 0 : row_slot + 1;
    }
    if (++cons_part == cpr) cons_part = 0;
    if (++cons_stage == kStages) {
      cons_stage = 0;
      cons_parity ^= 1u;
    }
    if (++nxt_part == cpr) {
      nxt_part = 0;
      nxt_row += gridDim.x;
    }
  }
  __syncthreads();  // every warp has left the loop (finished, or given up after a bounded wait)
  if (abort_flag) {
    // a copy did not complete in time: record the fault for hlo_device_faults(), wait (bounded) for
    // each stage's last copy, then mark this block's rows NaN so the failure also shows in the output
    if (tid == 0) record_fault(kFaultCopyTimeout);
    if (tid == 0)
      for (int st = 0; st < kStages; ++st)
        if (last_issued[st] >= 0)
          mbar_wait(smem_addr(&bar[st]), (uint32_t)((last_issued[st] / kStages) & 1));
    for (int64_t r = tid; r < my_rows; r += kStreamThreads)
      store_result(p.out, p.out_dt, map_index(p.omap, blockIdx.x + r * gridDim.x), __int_as_float(0x7FC00000));
  }
}

template <int IN_DT, int KIND>
static cudaError_t stream_dispatch(const RowReducePlan& p, cudaStream_t s, int ch) {
  auto launch = [&](auto kernel) -> cudaError_t {
    const size_t smem = (size_t)kStages * kChunkBytes;
    const int nb = kernel_blocks_per_sm((const void*)kernel, kStreamThreads, smem);
    int64_t grid = (int64_t)device_sm_count() * nb;
    if (grid > p.rows) grid = p.rows;
    const int cpr = (int)((p.len * dt_bytes(IN_DT) + kChunkBytes - 1) / kChunkBytes);
    kernel<<<(unsigned)grid, kStreamThreads, smem, s>>>(p, cpr);
    return cudaGetLastError();
  };
  const bool two_chunks = p.len * dt_bytes(IN_DT) <= 2 * (int64_t)kChunkBytes;
  if (ch == RC_EXP_BCAST_BF16 && IN_DT == BF16) {
    if (two_chunks && KIND == RED_ADD) return launch(row_stream_kernel<BF16, RC_EXP_BCAST_BF16, KIND, true>);
    return launch(row_stream_kernel<BF16, RC_EXP_BCAST_BF16, KIND, false>);
  }
  if (ch == RC_EXP) return launch(row_stream_kernel<IN_DT, RC_EXP, KIND, false>);
  return launch(row_stream_kernel<IN_DT, RC_NONE, KIND, false>);
}

// Row kernel for the runtime chain when the broadcast operand is per row or the vector path does
// not apply: scalar loads, any chain.
template <int IN_DT, int KIND>
__global__ void __launch_bounds__(kRowThreads) row_reduce_rt_kernel(RowReducePlan p) {
  __shared__ float red[32];
  __shared__ float4 s_lc[HLO_LOG_NC];
  __shared__ float2 s_le[HLO_LOG_NE];
  LogTab lt = global_log_tables();
  if (chain_has_log(p.chain)) {
    load_log_tables(s_lc, s_le);
    __syncthreads();
    lt = {s_lc, s_le};
  }
  const int64_t n_items = p.rows * p.split;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int64_t row = item / p.split, sg = item - row * p.split;
    const int64_t e0 = sg * p.seg, e1 = min(p.len, e0 + p.seg);
    const char* base = reinterpret_cast<const char*>(p.in) + row * p.len * dt_bytes(IN_DT);
    const int64_t rowb = p.bmode == BC_PERROW ? map_index(p.bmap, row) : 0;
    float acc = identity<KIND>();
    for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
      float t = load_as_f32(base, IN_DT, e);
      int64_t boff = p.bmode == BC_ROWVEC ? e : rowb;
      t = apply_chain_rt(p.chain, t, boff, lt);
      acc = combine<KIND>(acc, t);
    }
    acc = block_reduce<KIND>(acc, red);
    if (threadIdx.x == 0) {
      if (p.split > 1) p.ws[item] = acc;
      else store_result(p.out, p.out_dt, map_index(p.omap, row), combine<KIND>(p.init, acc));
    }
  }
}

// Short rows (at most 512 16-byte vectors): one warp per row, eight rows per block. Every lane requests
// its vectors before using any, and the warp combines with shuffles only: no block barrier, no shared
// memory, one wave for a few hundred rows.
constexpr int kWarpRowMaxVec = 512;
template <int IN_DT, int CH, int KIND>
__global__ void __launch_bounds__(256) row_warp_kernel(RowReducePlan p) {
  constexpr int V = IN_DT == F32 ? 4 : 8;
  constexpr int kU = 4;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= p.rows) return;
  const int64_t nvec = p.len / V;  // the row is whole 16-byte vectors
  const uint4* xv = reinterpret_cast<const uint4*>(p.in) + row * nvec;
  const LogTab lt = global_log_tables();
  const uint4 zero = make_uint4(0, 0, 0, 0);
  float acc = identity<KIND>();
  int64_t v = lane;
  for (; v + 32 * (kU - 1) < nvec; v += 32 * kU) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(x[u].x), "=r"(x[u].y), "=r"(x[u].z), "=r"(x[u].w)
                   : "l"(xv + v + 32 * u));
#pragma unroll
    for (int u = 0; u < kU; ++u) acc = row_vec<IN_DT, CH, KIND>(x[u], zero, acc, p.chain, lt);
  }
  for (; v < nvec; v += 32) acc = row_vec<IN_DT, CH, KIND>(__ldg(xv + v), zero, acc, p.chain, lt);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = combine<KIND>(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  if (lane == 0) store_result(p.out, p.out_dt, map_index(p.omap, row), combine<KIND>(p.init, acc));
}

template <int IN_DT, int KIND>
static cudaError_t row_dispatch(const RowReducePlan& p, cudaStream_t s, int ch, bool vec) {
  auto launch = [&](auto kernel) -> cudaError_t {
    const int nb = kernel_blocks_per_sm((const void*)kernel, kRowThreads, 0);
    int64_t grid = (int64_t)device_sm_count() * nb;
    const int64_t items = p.rows * p.split;
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    int threads = kRowThreads;
    // short rows (segments): fewer threads so that lanes are not idle
    const int64_t seg_len = p.split > 1 ? p.seg : p.len;
    int64_t work = vec ? (seg_len / (IN_DT == F32 ? 4 : 8)) : seg_len;
    while (threads > 64 && work <= threads / 2) threads >>= 1;
    kernel<<<(unsigned)grid, threads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.split <= 1) return e;
    int64_t cb = (p.rows + 255) / 256;
    if (cb > 1024) cb = 1024;
    row_split_combine_kernel<KIND><<<(unsigned)cb, 256, 0, s>>>(p);
    return cudaGetLastError();
  };
  constexpr int V = IN_DT == F32 ? 4 : 8;
  if (ch == RC_RT && p.bmode == BC_PERROW) return launch(row_reduce_rt_kernel<IN_DT, KIND>);
  if (vec && p.split <= 1 && (ch == RC_NONE || ch == RC_EXP) && p.len / V <= kWarpRowMaxVec) {
    const int64_t blocks = (p.rows + 7) / 8;
    if (blocks <= 0x7FFFFFFF) {
      if (ch == RC_NONE) row_warp_kernel<IN_DT, RC_NONE, KIND><<<(unsigned)blocks, 256, 0, s>>>(p);
      else row_warp_kernel<IN_DT, RC_EXP, KIND><<<(unsigned)blocks, 256, 0, s>>>(p);
      return cudaGetLastError();
    }
  }
  if (vec) {
    switch (ch) {
      case RC_NONE: return launch(row_reduce_kernel<IN_DT, V, RC_NONE, KIND>);
      case RC_EXP: return launch(row_reduce_kernel<IN_DT, V, RC_EXP, KIND>);
      case RC_EXP_BCAST_BF16:
        if (IN_DT == BF16) return launch(row_reduce_kernel<BF16, 8, RC_EXP_BCAST_BF16, KIND>);
        break;
      default: break;
    }
    return launch(row_reduce_rt_kernel<IN_DT, KIND>);
  }
  switch (ch) {
    case RC_NONE: return launch(row_reduce_kernel<IN_DT, 1, RC_NONE, KIND>);
    case RC_EXP: return launch(row_reduce_kernel<IN_DT, 1, RC_EXP, KIND>);
    default: return launch(row_reduce_rt_kernel<IN_DT, KIND>);
  }
}

static int classify_row_chain(const RowReducePlan& p) {
  const Chain& c = p.chain;
  if (c.n == 0) return RC_NONE;
  if (c.n == 1 && c.op[0] == OP_EXP) return RC_EXP;
  if (c.n == 2 && c.op[0] == OP_EXP && c.op[1] == OP_ADD_BCAST && c.dt == BF16 && c.bdt == BF16 &&
      c.round16 && p.bmode == BC_ROWVEC)
    return RC_EXP_BCAST_BF16;
  return RC_RT;
}

int64_t row_split_factor(int64_t rows, int64_t len, int eb) {
  // 512-thread blocks, four per SM: split while the rows fill less than half of those slots, into
  // segments of at least 32 KiB
  const int64_t slots = (int64_t)device_sm_count() * 4;
  if (rows <= 0 || rows * 2 > slots) return 1;
  const int64_t min_seg = 32768 / eb;
  int64_t split = (slots + rows - 1) / rows;
  const int64_t by_len = len / min_seg;
  if (split > by_len) split = by_len;
  return split > 1 ? split : 1;
}

cudaError_t launch_row_reduce(const RowReducePlan& p, cudaStream_t s) {
  const int eb = dt_bytes(p.in_dt);
  const int ch = classify_row_chain(p);
  // 16-byte vectors need 16-byte aligned rows (and broadcast vector, when streamed alongside)
  bool vec = ((uintptr_t)p.in % 16 == 0) && ((p.len * eb) % 16 == 0);
  if (ch == RC_EXP_BCAST_BF16) vec = vec && ((uintptr_t)p.chain.bptr % 16 == 0);
  if (ch == RC_RT) vec = false;
  // long rows on the vector path stream through the bulk-copy ring
  const bool stream = vec && ch != RC_RT && p.len * eb >= 8192 && p.rows >= 64 && p.split <= 1;
  if (stream) {
    if (p.in_dt == F32)
      return p.kind == RED_ADD ? stream_dispatch<F32, RED_ADD>(p, s, ch) : stream_dispatch<F32, RED_MAX>(p, s, ch);
    if (p.in_dt == BF16)
      return p.kind == RED_ADD ? stream_dispatch<BF16, RED_ADD>(p, s, ch) : stream_dispatch<BF16, RED_MAX>(p, s, ch);
    return p.kind == RED_ADD ? stream_dispatch<F16, RED_ADD>(p, s, ch) : stream_dispatch<F16, RED_MAX>(p, s, ch);
  }
  if (p.in_dt == F32)
    return p.kind == RED_ADD ? row_dispatch<F32, RED_ADD>(p, s, ch, vec) : row_dispatch<F32, RED_MAX>(p, s, ch, vec);
  if (p.in_dt == BF16)
    return p.kind == RED_ADD ? row_dispatch<BF16, RED_ADD>(p, s, ch, vec) : row_dispatch<BF16, RED_MAX>(p, s, ch, vec);
  return p.kind == RED_ADD ? row_dispatch<F16, RED_ADD>(p, s, ch, vec) : row_dispatch<F16, RED_MAX>(p, s, ch, vec);
}

// ---- device faults -------------------------------------------------------------------------------
// One block waits, with a short bound, on an mbarrier that nothing completes: the bounded wait of the
// streaming kernels runs out and records the same fault bit they record, so that the reporting path
// can be checked without a failing copy.
__global__ void wait_selftest_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_addr(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait(smem_addr(&bar), 0, limit)) record_fault(kFaultCopyTimeout);
}

cudaError_t launch_wait_selftest(cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(2000000LL);  // ~1 ms
  return cudaGetLastError();
}


// ---- column reduce --------------------------------------------------------------------------------
constexpr int kColCluster = 8;
constexpr int kColWarps = 8;
constexpr int kColUnroll = 8;

// Block (x = column block * kColCluster + slab, y = a). Each lane owns VEC consecutive columns.
template <int IN_DT, int VEC, int KIND, bool RT>
__global__ void __launch_bounds__(kColWarps * 32) col_reduce_kernel(ColReducePlan p, int64_t rows_per_slab) {
  __shared__ float part[kColWarps][32 * VEC];
  __shared__ float4 s_lc[HLO_LOG_NC];
  __shared__ float2 s_le[HLO_LOG_NE];
  cg::cluster_group cluster = cg::this_cluster();
  LogTab lt = global_log_tables();
  if (RT && chain_has_log(p.chain)) {
    load_log_tables(s_lc, s_le);
    __syncthreads();
    lt = {s_lc, s_le};
  }
  const int slab = (int)cluster.block_rank();
  const int64_t colblock = blockIdx.x / kColCluster;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t col0 = (colblock * 32 + lane) * VEC;  // first column of this lane
  const int eb = dt_bytes(IN_DT);
  const int64_t B = p.b;
  const char* base = reinterpret_cast<const char*>(p.in) + (int64_t)blockIdx.y * p.r * B * eb;
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = identity<KIND>();
  const int64_t r0 = slab * rows_per_slab;
  const int64_t r1 = min(r0 + rows_per_slab, p.r);
  const bool active = col0 < B;
  if (active) {
    if (VEC > 1) {
      int64_t r = r0 + warp;
      for (; r + (kColUnroll - 1) * kColWarps < r1; r += kColUnroll * kColWarps) {
        uint4 x[kColUnroll];
#pragma unroll
        for (int u = 0; u < kColUnroll; ++u) {
          const uint4* ptr = reinterpret_cast<const uint4*>(base + ((r + u * kColWarps) * B + col0) * eb);
          asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(x[u].x), "=r"(x[u].y), "=r"(x[u].z), "=r"(x[u].w)
                       : "l"(ptr));
        }
#pragma unroll
        for (int u = 0; u < kColUnroll; ++u) {
          const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (IN_DT == F32) {
              float t = __uint_as_float(w[i]);
              if (RT) t = apply_chain_rt(p.chain, t, 0, lt);
              acc[i] = combine<KIND>(acc[i], t);
            } else {
              float lo = IN_DT == BF16 ? bf16_bits_to_f32(w[i] & 0xFFFFu) : f16_bits_to_f32((uint16_t)(w[i] & 0xFFFFu));
              float hi = IN_DT == BF16 ? __uint_as_float(w[i] & 0xFFFF0000u) : f16_bits_to_f32((uint16_t)(w[i] >> 16));
              if (RT) {
                lo = apply_chain_rt(p.chain, lo, 0, lt);
                hi = apply_chain_rt(p.chain, hi, 0, lt);
              }
              acc[2 * i] = combine<KIND>(acc[2 * i], lo);
              acc[2 * i + 1] = combine<KIND>(acc[2 * i + 1], hi);
            }
          }
        }
      }
      for (; r < r1; r += kColWarps) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(base + (r * B + col0) * eb));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (IN_DT == F32) {
            float t = __uint_as_float(w[i]);
            if (RT) t = apply_chain_rt(p.chain, t, 0, lt);
            acc[i] = combine<KIND>(acc[i], t);
          } else {
            float lo = IN_DT == BF16 ? bf16_bits_to_f32(w[i] & 0xFFFFu) : f16_bits_to_f32((uint16_t)(w[i] & 0xFFFFu));
            float hi = IN_DT == BF16 ? __uint_as_float(w[i] & 0xFFFF0000u) : f16_bits_to_f32((uint16_t)(w[i] >> 16));
            if (RT) {
              lo = apply_chain_rt(p.chain, lo, 0, lt);
              hi = apply_chain_rt(p.chain, hi, 0, lt);
            }
            acc[2 * i] = combine<KIND>(acc[2 * i], lo);
            acc[2 * i + 1] = combine<KIND>(acc[2 * i + 1], hi);
          }
        }
      }
    } else {
      for (int64_t r = r0 + warp; r < r1; r += kColWarps) {
        float t = load_as_f32(base, IN_DT, r * B + col0);
        if (RT) t = apply_chain_rt(p.chain, t, 0, lt);
        acc[0] = combine<KIND>(acc[0], t);
      }
    }
  }
  // combine the warps of this block
#pragma unroll
  for (int i = 0; i < VEC; ++i) part[warp][lane * VEC + i] = acc[i];
  __syncthreads();
  for (int c = threadIdx.x; c < 32 * VEC; c += blockDim.x) {
    float v = part[0][c];
    for (int w = 1; w < kColWarps; ++w) v = combine<KIND>(v, part[w][c]);
    part[0][c] = v;
  }
  // combine the slabs of the cluster in rank order (deterministic), in block rank 0
  cluster.sync();
  if (slab == 0) {
    for (int c = threadIdx.x; c < 32 * VEC; c += blockDim.x) {
      float v = part[0][c];
      for (int q = 1; q < kColCluster; ++q) {
        const float* peer = cluster.map_shared_rank(&part[0][0], q);
        v = combine<KIND>(v, peer[c]);
      }
      const int64_t col = colblock * 32 * VEC + c;
      if (col < B) {
        const int64_t k = (int64_t)blockIdx.y * B + col;
        store_result(p.out, p.out_dt, map_index(p.omap, k), combine<KIND>(p.init, v));
      }
    }
  }
  cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

template <int IN_DT, int VEC, int KIND, bool RT>
static cudaError_t col_launch(const ColReducePlan& p, cudaStream_t s) {
  const int64_t ncb = (p.b + 32 * VEC - 1) / (32 * VEC);
  const int64_t rows_per_slab = (p.r + kColCluster - 1) / kColCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ncb * kColCluster), (unsigned)p.a, 1);
  cfg.blockDim = dim3(kColWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kColCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, col_reduce_kernel<IN_DT, VEC, KIND, RT>, p, rows_per_slab);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int IN_DT, int KIND>
static cudaError_t col_dispatch(const ColReducePlan& p, cudaStream_t s) {
  constexpr int V = IN_DT == F32 ? 4 : 8;
  const bool rt = p.chain.n > 0;
  const bool vec = ((uintptr_t)p.in % 16 == 0) && ((p.b * dt_bytes(IN_DT)) % 16 == 0);
  if (vec) return rt ? col_launch<IN_DT, V, KIND, true>(p, s) : col_launch<IN_DT, V, KIND, false>(p, s);
  return rt ? col_launch<IN_DT, 1, KIND, true>(p, s) : col_launch<IN_DT, 1, KIND, false>(p, s);
}

cudaError_t launch_col_reduce(const ColReducePlan& p, cudaStream_t s) {
  if (p.in_dt == F32) return p.kind == RED_ADD ? col_dispatch<F32, RED_ADD>(p, s) : col_dispatch<F32, RED_MAX>(p, s);
  if (p.in_dt == BF16) return p.kind == RED_ADD ? col_dispatch<BF16, RED_ADD>(p, s) : col_dispatch<BF16, RED_MAX>(p, s);
  return p.kind == RED_ADD ? col_dispatch<F16, RED_ADD>(p, s) : col_dispatch<F16, RED_MAX>(p, s);
}

// ---- general reduce -------------------------------------------------------------------------------
// Sums are formed in chunks of 256 terms so that the f32 error stays near (256 + n/256) ulp.
__global__ void __launch_bounds__(256) gen_reduce_kernel(GenReducePlan p) {
  const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= p.n_out) return;
  const LogTab lt = global_log_tables();
  // decompose o over the kept axes in output physical order
  int64_t rem = o, base = 0, bbase = 0;
  for (int j = p.nk - 1; j >= 0; --j) {
    int64_t i = rem % p.kdim_size[j];
    rem /= p.kdim_size[j];
    base += i * p.kdim_in_stride[j];
    bbase += i * p.chain.bstride[p.kdim_logical[j]];
  }
  float total = p.kind == RED_ADD ? 0.f : __int_as_float(0xFF800000);
  float chunk = total;
  int64_t ridx[kMaxRank];
  for (int j = 0; j < p.nr; ++j) ridx[j] = 0;
  for (int64_t t = 0; t < p.n_red; ++t) {
    int64_t off = base, boff = bbase;
    for (int j = 0; j < p.nr; ++j) {
      off += ridx[j] * p.rdim_in_stride[j];
      boff += ridx[j] * p.chain.bstride[p.rdim_logical[j]];
    }
    float v = apply_chain_rt(p.chain, load_as_f32(p.in, p.in_dt, off), boff, lt);
    chunk = combine_rt(p.kind, chunk, v);
    if ((t & 255) == 255) {
      total = combine_rt(p.kind, total, chunk);
      chunk = p.kind == RED_ADD ? 0.f : __int_as_float(0xFF800000);
    }
    for (int j = p.nr - 1; j >= 0; --j) {  // odometer over the reduced axes, minor fastest
      if (++ridx[j] < p.rdim_size[j]) break;
      ridx[j] = 0;
    }
  }
  total = combine_rt(p.kind, total, chunk);
  store_result(p.out, p.out_dt, o, combine_rt(p.kind, p.init, total));
}

cudaError_t launch_gen_reduce(const GenReducePlan& p, cudaStream_t s) {
  if (p.n_out == 0) return cudaSuccess;
  const int64_t blocks = (p.n_out + 255) / 256;
  gen_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

__global__ void fill_kernel(void* out, int dt, int64_t n, float value) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    store_from_f32(out, dt, i, value);
}

cudaError_t launch_fill(void* out, int dt, int64_t n, float value, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_kernel<<<(unsigned)blocks, 256, 0, s>>>(out, dt, n, value);
  return cudaGetLastError();
}

}  // namespace hlo
