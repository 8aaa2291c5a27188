// Self-add transpose hero kernels: out = f(p) + transpose(f(p)) for an n x n array ("XLA:GPU Emitters",
// sections "Partitioning" -- the param -> log -> {transpose, add} graph, where the log is evaluated
// once per element -- and "Transpose emitter": coalesced reads into a shared-memory tile, a barrier,
// coalesced writes out of it). A block owns a tile pair (I,J), (J,I): it reads both once, applies the
// prologue f once per element, and writes both output tiles.
//
//  selfadd_tma_kernel   -- rows on 16-byte boundaries: 2-D tensor copies into a ring of shared-memory
//                          stages, the prologue computed in place, transposed 16-byte stores.
//  selfadd_pair_kernel  -- any row alignment (and aligned rows when no tensor map can be made): padded
//                          shared tiles, 16-byte or scalar global accesses.
#include "async_copy.cuh"
#include "device_common.cuh"

namespace hlo {

// ---------------------------------------------------------------------------------------------
// pair-tile self-add transpose
// ---------------------------------------------------------------------------------------------
constexpr int kT = 64;        // tile edge (elements)
constexpr int kTP = kT + 1;   // padded pitch: transposed stores and row reads hit 32 distinct banks
constexpr int kPairThreads = 256;

enum PairChain : int { PC_NONE = 0, PC_LOG = 1, PC_RT = 2 };

// Maps a pair index to (I, J), I < J, enumerating row by row: a single-precision estimate from the
// quadratic formula, then exact integer correction. Only 32-bit integer <-> float conversions are used
// (64-bit ones run on the FP64 pipe, a slow unit on this part); the launcher guarantees that the pair
// count fits in 31 bits.
__device__ __forceinline__ void pair_of(int64_t item, int64_t nt, int64_t& I, int64_t& J) {
  const float b = 2.0f * (float)(int)nt - 1.0f;
  const float disc = fmaxf(b * b - 8.0f * (float)(int)item, 0.0f);
  int64_t i = (int)((b - sqrtf(disc)) * 0.5f);
  i = i < 0 ? 0 : (i > nt - 2 ? nt - 2 : i);
  auto start = [nt](int64_t r) { return r * (nt - 1) - ((r * (r - 1)) >> 1); };
  while (i > 0 && start(i) > item) --i;
  while (start(i + 1) <= item) ++i;
  I = i;
  J = i + 1 + (item - start(i));
}

template <int CH>
__device__ __forceinline__ float pair_pro(float v, const Chain& c, const LogTab& lt) {
  if (CH == PC_LOG) return cr_logf(v, lt.c, lt.e);
  if (CH == PC_RT) return apply_chain_rt(c, v, 0, lt);
  return v;
}

// Thread mapping inside a 64 x 64 tile: slot k (0..3) of warp w covers rows 4*rg .. 4*rg+3, columns
// 32*h .. 32*h+31, with 8 lanes (16 bytes each) per 128-byte row segment. A lane owns row
// r = 4*rg + lane/8 and columns c .. c+3, c = 32*h + 4*(lane%8).
__device__ __forceinline__ void pair_slot(int k, int& r, int& c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int s = warp * 4 + k;
  r = 4 * (s >> 1) + (lane >> 3);
  c = 32 * (s & 1) + 4 * (lane & 7);
}

// Shared state of the pair kernel's log: the two-pass tables and the list of elements whose rounding
// the first pass left open (their slot offsets; the slot holds the input meanwhile).
constexpr int kRedoCap = 2048;
struct PairShared {
  float l1_inv[32], l1_hi[32], l1_lo[32];
  int redo_count;
  uint16_t redo[kRedoCap];
};

// Loads this thread's 16 elements of tile (TI, TJ), applies the prologue and stores the results
// transposed: dst[col * kTP + row]. With kTP = 65 the 32 lanes of a store hit 32 distinct banks.
// For log, the first pass (two elements per f32x2 instruction) settles ~98% of the elements; the
// others are parked (input value in the slot) on the block's redo list, or in the thread's own
// spill mask if the list is full, and settled after the barrier.
template <int CH, bool VEC>
__device__ __forceinline__ void pair_load(const float* __restrict__ in, int64_t n, int64_t TI, int64_t TJ,
                                          const int (&toff)[4], float* dst, int dst_base, const Chain& c,
                                          const LogTab& lt, PairShared& ps, uint32_t& spill) {
  float4 v[4];
  const float* tile = in + TI * kT * n + TJ * kT;          // element (0, 0) of the tile
  const bool full = (TI + 1) * kT <= n && (TJ + 1) * kT <= n;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int r, col;
    pair_slot(k, r, col);
    const int64_t gr = TI * kT + r, gc = TJ * kT + col;
    if (VEC) {
      if (full || (gr < n && gc < n)) {
        const float4* src = reinterpret_cast<const float4*>(tile + toff[k]);
        asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v[k].x), "=f"(v[k].y), "=f"(v[k].z), "=f"(v[k].w)
                     : "l"(src));
      } else {
        v[k] = make_float4(1.f, 1.f, 1.f, 1.f);
      }
    } else {
      float* o = &v[k].x;
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = (gr < n && gc + q < n) ? in[gr * n + gc + q] : 1.f;
    }
  }
  uint32_t redo = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int r, col;
    pair_slot(k, r, col);
    float y[4];
    if (CH == PC_LOG) {
      bool ok[4];
      cr_logf_first2(v[k].x, v[k].y, ps.l1_inv, ps.l1_hi, ps.l1_lo, y[0], y[1], ok[0], ok[1]);
      cr_logf_first2(v[k].z, v[k].w, ps.l1_inv, ps.l1_hi, ps.l1_lo, y[2], y[3], ok[2], ok[3]);
      const float* xi = &v[k].x;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        redo |= (ok[q] ? 0u : 1u) << (4 * k + q);
        y[q] = ok[q] ? y[q] : xi[q];  // park the input of an open element in its slot
      }
    } else {
      const float* xi = &v[k].x;
#pragma unroll
      for (int q = 0; q < 4; ++q) y[q] = pair_pro<CH>(xi[q], c, lt);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[(col + q) * kTP + r] = y[q];
  }
  if (CH == PC_LOG) {
    // append the open elements to the block list: one atomic per warp
    const int lane = threadIdx.x & 31;
    const int cnt = __popc(redo);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total) {
      int base = 0;
      if (lane == 31) base = atomicAdd(&ps.redo_count, total);
      base = __shfl_sync(0xffffffffu, base, 31);
      int pos = base + incl - cnt;
      uint32_t m = redo;
      while (m) {
        const int e = __ffs(m) - 1;
        m &= m - 1;
        int r, col;
        pair_slot(e >> 2, r, col);
        const int off = dst_base + (col + (e & 3)) * kTP + r;
        if (pos < kRedoCap) ps.redo[pos] = (uint16_t)off;
        else spill |= 1u << (e + (dst_base ? 16 : 0));
        ++pos;
      }
    }
  }
}

// Settles the elements the first pass left open -- the block's list, then this thread's spills --
// from the input parked in their slot.
__device__ __forceinline__ void pair_settle(float* tiles, PairShared& ps, uint32_t spill, const LogTab& lt) {
  const int cnt = min(ps.redo_count, kRedoCap);
  for (int j = threadIdx.x; j < cnt; j += kPairThreads) {
    float* slot = tiles + ps.redo[j];
    *slot = cr_logf(*slot, lt.c, lt.e);
  }
  while (spill) {
    const int e = __ffs(spill) - 1;
    spill &= spill - 1;
    int r, col;
    pair_slot((e & 15) >> 2, r, col);
    float* slot = tiles + ((e >= 16) ? kT * kTP : 0) + (col + (e & 3)) * kTP + r;
    *slot = cr_logf(*slot, lt.c, lt.e);
  }
}

// Writes this thread's 16 elements of output tile (TI, TJ) = own[r][c] + other[c][r], where ownT and
// otherT hold the two tiles transposed (so own[r][c] = ownT[c][r], other[c][r] = otherT[r][c]), then
// the epilogue. Both reads hit 32 distinct banks per warp.
template <bool VEC>
__device__ __forceinline__ void pair_store(float* __restrict__ out, int64_t n, int64_t TI, int64_t TJ,
                                           const int (&toff)[4], const float* ownT, const float* otherT,
                                           const Chain& epi, const LogTab& lt) {
  float* tile = out + TI * kT * n + TJ * kT;
  const bool full = (TI + 1) * kT <= n && (TJ + 1) * kT <= n;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int r, col;
    pair_slot(k, r, col);
    const float* t = otherT + r * kTP + col;
    const float* o = ownT + col * kTP + r;
    float4 v;
    v.x = __fadd_rn(o[0 * kTP], t[0]);
    v.y = __fadd_rn(o[1 * kTP], t[1]);
    v.z = __fadd_rn(o[2 * kTP], t[2]);
    v.w = __fadd_rn(o[3 * kTP], t[3]);
    if (epi.n) {
      v.x = apply_chain_rt(epi, v.x, 0, lt);
      v.y = apply_chain_rt(epi, v.y, 0, lt);
      v.z = apply_chain_rt(epi, v.z, 0, lt);
      v.w = apply_chain_rt(epi, v.w, 0, lt);
    }
    const int64_t gr = TI * kT + r, gc = TJ * kT + col;
    if (VEC) {
      if (full || (gr < n && gc < n)) *reinterpret_cast<float4*>(tile + toff[k]) = v;
    } else {
      const float* pv = &v.x;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (gr < n && gc + q < n) out[gr * n + gc + q] = pv[q];
    }
  }
}

template <int CH, bool VEC>
__global__ void __launch_bounds__(kPairThreads, 4)
    selfadd_pair_kernel(SelfAddPlan p, int64_t nt, int64_t n_off, int64_t n_items) {
  extern __shared__ float4 smem_f4[];
  float4* s_lc = smem_f4;
  float2* s_le = reinterpret_cast<float2*>(s_lc + HLO_LOG_NC);
  float* ta = reinterpret_cast<float*>(s_le + HLO_LOG_NE);  // tile (I,J) after the prologue, transposed
  float* tb = ta + kT * kTP;                                 // tile (J,I) after the prologue, transposed
  PairShared& ps = *reinterpret_cast<PairShared*>(tb + kT * kTP);
  load_log_tables(s_lc, s_le);
  load_log1_tables(ps.l1_inv, ps.l1_hi, ps.l1_lo);
  if (threadIdx.x == 0) ps.redo_count = 0;
  __syncthreads();
  const LogTab lt = {s_lc, s_le};
  const float* in = reinterpret_cast<const float*>(p.in);
  float* out = reinterpret_cast<float*>(p.out);
  int toff[4];  // this thread's in-tile element offsets (row * n + column); 64 * n < 2^31 always holds
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int r, col;
    pair_slot(k, r, col);
    toff[k] = r * (int)p.n + col;
  }
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    int64_t I, J;
    if (item < n_off) {
      pair_of(item, nt, I, J);
    } else {
      I = J = item - n_off;
    }
    uint32_t spill = 0;
    pair_load<CH, VEC>(in, p.n, I, J, toff, ta, 0, p.pro, lt, ps, spill);
    if (I != J) pair_load<CH, VEC>(in, p.n, J, I, toff, tb, kT * kTP, p.pro, lt, ps, spill);
    __syncthreads();
    if (CH == PC_LOG) {
      if (ps.redo_count) {  // uniform: every thread reads the same count after the barrier
        pair_settle(ta, ps, spill, lt);
        __syncthreads();
      }
    }
    if (I != J) {
      pair_store<VEC>(out, p.n, I, J, toff, ta, tb, p.epi, lt);  // out(I,J) = A + B^T
      pair_store<VEC>(out, p.n, J, I, toff, tb, ta, p.epi, lt);  // out(J,I) = B + A^T
    } else {
      pair_store<VEC>(out, p.n, I, I, toff, ta, ta, p.epi, lt);
    }
    if (threadIdx.x == 0) ps.redo_count = 0;  // nobody reads it again before the barrier below
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------------
// Register-blocked thread mapping of the tensor-copy kernel below (rows on 16-byte boundaries).
// Thread t owns the 4 x 4 block (bi, bj) = (t / 16, t % 16) of each 64 x 64 tile:
//   1. it reads its block of tile A = (I,J) and of tile B = (J,I) (four 16-byte reads each), applies
//      the prologue in registers and writes the blocks back, 16-byte chunk c of row r at chunk
//      c ^ ((r / 4) % 8) of that row;
//   2. the block settles the log elements the first pass left open (one block list, a barrier, then
//      one open element per thread);
//   3. after a barrier it reads its block of A and block (bj, bi) of B, both as four 16-byte reads that
//      hit 32 distinct banks per quarter-warp, transposes the latter in registers and writes block
//      (bi, bj) of out(I,J) = A + B^T with four 16-byte stores; then out(J,I) = B + A^T alike.
// Every element is read once, goes through the prologue once, is written to and read from shared
// memory with one 16-byte access each way, and is stored once.
// ---------------------------------------------------------------------------------------------
constexpr int kBlockList = 512;  // open log elements a block settles together per item (about 150 expected)

__device__ __forceinline__ float comp(const float4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

__device__ __forceinline__ void item_pair(int64_t item, int64_t nt, int64_t n_off, int64_t& I, int64_t& J) {
  if (item < n_off) {
    pair_of(item, nt, I, J);
  } else {
    I = J = item - n_off;
  }
}

// Log of a block's four rows in registers: settled elements take their log, open ones keep their input
// and set bit 4k+q (+ shift) of `open`.
__device__ __forceinline__ void block_log(float4 (&v)[4], const float* tinv, const float* thi, const float* tlo,
                                          uint32_t& open, int shift) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float y[4];
    bool ok[4];
    cr_logf_first2(v[k].x, v[k].y, tinv, thi, tlo, y[0], y[1], ok[0], ok[1]);
    cr_logf_first2(v[k].z, v[k].w, tinv, thi, tlo, y[2], y[3], ok[2], ok[3]);
    v[k].x = ok[0] ? y[0] : v[k].x;
    v[k].y = ok[1] ? y[1] : v[k].y;
    v[k].z = ok[2] ? y[2] : v[k].z;
    v[k].w = ok[3] ? y[3] : v[k].w;
    open |= ((ok[0] ? 0u : 1u) | (ok[1] ? 0u : 2u) | (ok[2] ? 0u : 4u) | (ok[3] ? 0u : 8u)) << (4 * k + shift);
  }
}

// Writes block (bi, bj) of an output tile: row k = a[k] + column k of b (b holds the other tile's
// block (bj, bi) row by row), then the epilogue. `rows` = rows of the tile left from row 4*bi.
template <bool EPI>
__device__ __forceinline__ void block_store(float* dst, int64_t n, const float4 (&a)[4], const float4 (&b)[4],
                                            int64_t rows, bool cols_ok, const Chain& epi, const LogTab& lt) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float4 v;
    v.x = __fadd_rn(a[k].x, comp(b[0], k));
    v.y = __fadd_rn(a[k].y, comp(b[1], k));
    v.z = __fadd_rn(a[k].z, comp(b[2], k));
    v.w = __fadd_rn(a[k].w, comp(b[3], k));
    if (EPI) {
      v.x = apply_chain_rt(epi, v.x, 0, lt);
      v.y = apply_chain_rt(epi, v.y, 0, lt);
      v.z = apply_chain_rt(epi, v.z, 0, lt);
      v.w = apply_chain_rt(epi, v.w, 0, lt);
    }
    if (cols_ok && k < rows) *reinterpret_cast<float4*>(dst + k * n) = v;
  }
}

// ---------------------------------------------------------------------------------------------
// Tensor-copy pair kernel (the path for rows on 16-byte boundaries when the driver's tensor-map
// encoder is available), with the register-blocked mapping above. The raw input arrives by 2-D tensor
// copies (cp.async.bulk.tensor, one
// 64 x 64 box per tile) into a ring of NS shared-memory stages, and the prologue's results are
// written back into the stage they were read from:
//   wait for the stage's mbarrier; then per tile: 16-byte reads of the raw rows (a quarter warp reads
//   128 contiguous bytes), the prologue in registers, __syncwarp, 16-byte writes of the results to
//   the swizzled positions. A thread's swizzled chunk lies in its own four rows, which only its own
//   half warp reads, so the warp-level sync orders the in-place rewrite; then the block settles its
//   open log elements (a barrier between the list and the settling); block barrier; transposed reads,
//   add, 16-byte stores.
// After its stores each warp counts itself done with the stage; the last of the 8 warps refills the
// stage with the block's item j + NS at once (it also records the item's tile pair for the readers),
// so the copies run about NS - 1 items ahead of use.
// A bounded wait that runs out makes the whole block stop (the decision is made block-wide at the
// barrier), record kFaultCopyTimeout, wait (bounded) for its copies in flight and return.
// ---------------------------------------------------------------------------------------------
constexpr int kPairWarps = kPairThreads / 32;

// Item k of block b in the walk: round-robin (k * G + b) for the `full` = n_items / G whole rounds;
// the last, partial round goes to the blocks in reverse (G - 1 - b), so that the blocks that take an
// extra item are the ones whose last whole round held a (half-cost) diagonal item. -1 past the block's
// last item.
__device__ __forceinline__ int64_t walk_item(int64_t b, int64_t k, int64_t g, int64_t n_items, int64_t full) {
  if (k < full) return k * g + b;
  if (k > full) return -1;
  const int64_t it = full * g + (g - 1 - b);
  return it < n_items ? it : -1;
}

template <int NS>
struct TmaShared {
  uint16_t blist[kBlockList];  // stage slots of the item's open log elements
  int bcount[2];               // fill of the list, by item parity (one is cleared while the other fills)
  int done[NS];            // warps done with the stage's current item
  int2 ij[NS];             // tile pair (I, J) of the stage's current item
  uint64_t full[NS];
};

template <int NS>
static size_t tma_smem_bytes() {
  return 128 /* alignment slack */ + (size_t)NS * 2 * kT * kT * sizeof(float) + HLO_LOG_NC * sizeof(float4) +
         HLO_LOG_NE * sizeof(float2) + sizeof(TmaShared<NS>);
}

// Prologue of one raw tile of the stage, written back in place (swizzled); open log elements keep
// their input and set their bits in `open` (from bit `shift`). `l1` is the first-pass log table in
// static shared memory.
template <int CH>
__device__ __forceinline__ void tma_tile_prologue(float* tile, int raw, int own, const SelfAddPlan& p, const LogTab& lt,
                                                  const float (&l1)[96], uint32_t& open, int shift) {
  float4 v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = *reinterpret_cast<const float4*>(tile + raw + k * kT);
  if (CH == PC_LOG) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float4 y;
      const uint32_t ok = cr_logf_first4(v[k], l1, y);
      v[k].x = (ok & 1u) ? y.x : v[k].x;  // an open element keeps its input in its slot
      v[k].y = (ok & 2u) ? y.y : v[k].y;
      v[k].z = (ok & 4u) ? y.z : v[k].z;
      v[k].w = (ok & 8u) ? y.w : v[k].w;
      open |= (~ok & 15u) << (4 * k + shift);
    }
  } else if (CH == PC_RT) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k].x = pair_pro<CH>(v[k].x, p.pro, lt);
      v[k].y = pair_pro<CH>(v[k].y, p.pro, lt);
      v[k].z = pair_pro<CH>(v[k].z, p.pro, lt);
      v[k].w = pair_pro<CH>(v[k].w, p.pro, lt);
    }
  }
  __syncwarp();  // the half warp owning these rows has read them
#pragma unroll
  for (int k = 0; k < 4; ++k) *reinterpret_cast<float4*>(tile + own + k * kT) = v[k];
}

// Settles the block's open log elements of item j in the stage (their slots hold the input): each lane
// with open elements reserves room in the block's list with one shared atomic, a block barrier, then
// the list is shared out one element per thread (one correctly rounded log each, about 150 of them on
// U(0.5, 2) inputs: five warps' worth instead of a round in each of the eight warps), and a lane whose
// elements did not fit settles the rest itself. The list's count alternates by item parity: the count
// of item j + 1 is cleared here, after every thread has added to item j's and read item j - 1's.
__device__ __forceinline__ void block_settle_list(uint32_t open, float* tiles, int own, uint16_t* bl, int* bcount,
                                                  int64_t j, const LogTab& lt) {
  const int cnt = __popc(open);
  int pos = cnt ? atomicAdd(&bcount[j & 1], cnt) : 0;
  while (open && pos < kBlockList) {
    const int b = __ffs(open) - 1;
    open &= open - 1;
    bl[pos++] = (uint16_t)((b >> 4) * (kT * kT) + own + ((b >> 2) & 3) * kT + (b & 3));
  }
  __syncthreads();  // the list and the parked inputs are visible to the whole block
  const int total = min(bcount[j & 1], kBlockList);
  if (threadIdx.x == 0) bcount[(j + 1) & 1] = 0;
  for (int q = threadIdx.x; q < total; q += kPairThreads) {
    float* sl = tiles + bl[q];
    *sl = cr_logf(*sl, lt.c, lt.e);
  }
  while (open) {
    const int b = __ffs(open) - 1;
    open &= open - 1;
    float* sl = tiles + (b >> 4) * (kT * kT) + own + ((b >> 2) & 3) * kT + (b & 3);
    *sl = cr_logf(*sl, lt.c, lt.e);
  }
}

template <int CH, bool EPI, int NS>
__global__ void __launch_bounds__(kPairThreads, NS == 2 ? 3 : 2)
    selfadd_tma_kernel(const __grid_constant__ CUtensorMap tmap, SelfAddPlan p, int64_t nt, int64_t n_off,
                       int64_t n_items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  float* stage = reinterpret_cast<float*>(base);              // [NS][2][64 * 64]: tile (I,J), tile (J,I)
  float4* s_lc = reinterpret_cast<float4*>(stage + NS * 2 * kT * kT);
  float2* s_le = reinterpret_cast<float2*>(s_lc + HLO_LOG_NC);
  TmaShared<NS>& ts = *reinterpret_cast<TmaShared<NS>*>(s_le + HLO_LOG_NE);
  __shared__ float l1[96];  // first-pass log table (inv_c, log(c)_hi, log(c)_lo), at a static address
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t full = n_items / gridDim.x;  // whole rounds of the walk (one division per thread)
  // copies item `it` (walk position j) into stage j % NS and records its tile pair there
  // The tile pairs of the block's items, worked out 64 walk positions at a time (chunk c: positions
  // 64c .. 64c + 63, in set c % 2) by 64 threads, so that a refill does no index arithmetic. Chunk c + 1
  // is planned at position 64c, before that item's barrier; the refills reading chunk c - 1 (the other
  // use of its set) all come before the previous item's barrier ends.
  __shared__ int2 s_pairs[2][64];
  auto plan_pairs = [&](int64_t c, int t) {  // thread t of 64 plans position 64c + t
    const int64_t it = walk_item(blockIdx.x, 64 * c + t, gridDim.x, n_items, full);
    int64_t I = -1, J = -1;
    if (it >= 0) item_pair(it, nt, n_off, I, J);
    s_pairs[c & 1][t] = make_int2((int)I, (int)J);
  };
  auto issue = [&](int64_t I, int64_t J, int64_t j) {
    const int st = (int)(j % NS);
    ts.ij[st] = make_int2((int)I, (int)J);
    const uint32_t bar = smem_addr(&ts.full[st]);
    float* dst = stage + st * 2 * kT * kT;
    mbar_arrive_expect_tx(bar, (I != J ? 2u : 1u) * kT * kT * (uint32_t)sizeof(float));
    tma_load_2d(dst, &tmap, (int32_t)(J * kT), (int32_t)(I * kT), bar);                      // tile (I, J)
    if (I != J) tma_load_2d(dst + kT * kT, &tmap, (int32_t)(I * kT), (int32_t)(J * kT), bar);  // tile (J, I)
  };
  if (tid == 0) {
    prefetch_tensor_map(&tmap);
    for (int st = 0; st < NS; ++st) {
      mbar_init(smem_addr(&ts.full[st]), 1);
      ts.done[st] = 0;
    }
    ts.bcount[0] = ts.bcount[1] = 0;
    fence_mbar_init();
    for (int64_t j = 0; j < NS; ++j) {
      const int64_t it = walk_item(blockIdx.x, j, gridDim.x, n_items, full);
      int64_t I, J;
      if (it >= 0) {
        item_pair(it, nt, n_off, I, J);
        issue(I, J, j);
      }
    }
  }
  load_log_tables(s_lc, s_le);
  load_log1_tables(l1, l1 + 32, l1 + 64);
  if (tid < 128) plan_pairs(tid >> 6, tid & 63);  // chunks 0 and 1
  __syncthreads();
  const LogTab lt = {s_lc, s_le};
  float* out = reinterpret_cast<float*>(p.out);
  const int64_t n = p.n;
  const int bi = tid >> 4, bj = tid & 15;
  const int own = 4 * bi * kT + ((bj ^ (bi & 7)) << 2);  // row 4*bi, chunk bj (swizzled)
  const int oth = 4 * bj * kT + ((bi ^ (bj & 7)) << 2);  // row 4*bj, chunk bi (swizzled)
  const int raw = 4 * bi * kT + 4 * bj;                  // row 4*bi, columns 4*bj.. of a raw tile
  const int64_t goff = 4 * bi * n + 4 * bj;
  int64_t j = 0;
  for (;; ++j) {
    const int64_t item = walk_item(blockIdx.x, j, gridDim.x, n_items, full);
    if (item < 0) break;
    if ((j & 63) == 0 && j > 0 && tid < 64) plan_pairs((j >> 6) + 1, tid);
    const int st = (int)(j % NS);
    const bool arrived = mbar_wait(smem_addr(&ts.full[st]), (uint32_t)((j / NS) & 1));
    const int2 ij = ts.ij[st];
    const int64_t I = ij.x, J = ij.y;
    const bool two = I != J;
    float* ta = stage + st * 2 * kT * kT;
    float* tb = ta + kT * kT;
    uint32_t open = 0;
    tma_tile_prologue<CH>(ta, raw, own, p, lt, l1, open, 0);
    if (two) tma_tile_prologue<CH>(tb, raw, own, p, lt, l1, open, 16);
    if (CH == PC_LOG) block_settle_list(open, ta, own, ts.blist, ts.bcount, j, lt);
    // every tile of item j is complete
    if (__syncthreads_or(arrived ? 0 : 1)) {
      // a copy did not arrive in time: record the fault, wait (bounded) for this block's copies still
      // in flight (items j .. j + NS - 1), leave the rest of its outputs unwritten and return
      if (tid == 0) {
        record_fault(kFaultCopyTimeout);
        for (int64_t q = j; q < j + NS && walk_item(blockIdx.x, q, gridDim.x, n_items, full) >= 0; ++q)
          mbar_wait(smem_addr(&ts.full[q % NS]), (uint32_t)((q / NS) & 1));
      }
      return;
    }
    const int64_t rows_a = n - I * kT - 4 * bi, rows_b = n - J * kT - 4 * bi;
    const bool ca = J * kT + 4 * bj < n, cb = I * kT + 4 * bj < n;
    {
      float4 a[4], b[4];
      const float* other = two ? tb : ta;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a[k] = *reinterpret_cast<const float4*>(ta + own + k * kT);
        b[k] = *reinterpret_cast<const float4*>(other + oth + k * kT);
      }
      block_store<EPI>(out + (I * kT) * n + J * kT + goff, n, a, b, rows_a, ca, p.epi, lt);  // out(I,J) = A + B^T
    }
    if (two) {
      float4 a[4], b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a[k] = *reinterpret_cast<const float4*>(tb + own + k * kT);
        b[k] = *reinterpret_cast<const float4*>(ta + oth + k * kT);
      }
      block_store<EPI>(out + (J * kT) * n + I * kT + goff, n, a, b, rows_b, cb, p.epi, lt);  // out(J,I) = B + A^T
    }
    // this warp's reads of the stage are complete (their values have been stored); the last warp out
    // refills the stage with item j + NS
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&ts.done[st], 1) == kPairWarps - 1) {
        ts.done[st] = 0;
        const int2 pr = s_pairs[((j + NS) >> 6) & 1][(j + NS) & 63];  // item j + NS, planned earlier
        if (pr.x >= 0) {
          fence_proxy_async();
          issue(pr.x, pr.y, j + NS);
        }
      }
    }
  }
}

// A 2-D f32 tensor map over the n x n row-major input with 64 x 64 boxes; false if it cannot be made.
static bool make_pair_tensor_map(const SelfAddPlan& p, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || p.n > (int64_t)INT32_MAX) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)p.n, (cuuint64_t)p.n};
  const cuuint64_t strides[1] = {(cuuint64_t)p.n * sizeof(float)};
  const cuuint32_t box[2] = {kT, kT};
  const cuuint32_t elem_strides[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(p.in), dims, strides, box, elem_strides,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef HLO_SELFADD_STAGES
#define HLO_SELFADD_STAGES 2
#endif
template <int CH, bool EPI>
static cudaError_t tma_launch(const SelfAddPlan& p, const CUtensorMap& map, cudaStream_t s) {
  constexpr int NS = HLO_SELFADD_STAGES;
  auto kernel = selfadd_tma_kernel<CH, EPI, NS>;
  const size_t smem = tma_smem_bytes<NS>();
  const int nb = kernel_blocks_per_sm((const void*)kernel, kPairThreads, smem);
  const int64_t nt = (p.n + kT - 1) / kT;
  const int64_t n_off = nt * (nt - 1) / 2;
  const int64_t n_items = n_off + nt;
  int64_t grid = (int64_t)device_sm_count() * nb;
  if (grid > n_items) grid = n_items;
  if (grid < 1) grid = 1;
  kernel<<<(unsigned)grid, kPairThreads, smem, s>>>(map, p, nt, n_off, n_items);
  return cudaGetLastError();
}


static size_t pair_smem_bytes() {
  return HLO_LOG_NC * sizeof(float4) + HLO_LOG_NE * sizeof(float2) + 2 * kT * kTP * sizeof(float) +
         sizeof(PairShared);
}

template <int CH, bool VEC>
static cudaError_t pair_launch(const SelfAddPlan& p, cudaStream_t s) {
  auto kernel = selfadd_pair_kernel<CH, VEC>;
  const size_t smem = pair_smem_bytes();
  const int nb = kernel_blocks_per_sm((const void*)kernel, kPairThreads, smem);
  const int64_t nt = (p.n + kT - 1) / kT;
  const int64_t n_off = nt * (nt - 1) / 2;
  const int64_t n_items = n_off + nt;
  int64_t grid = (int64_t)device_sm_count() * nb;
  if (grid > n_items) grid = n_items;
  if (grid < 1) grid = 1;
  kernel<<<(unsigned)grid, kPairThreads, smem, s>>>(p, nt, n_off, n_items);
  return cudaGetLastError();
}

cudaError_t launch_selfadd_transpose(const SelfAddPlan& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const bool vec = (p.n % 4 == 0) && ((uintptr_t)p.in % 16 == 0) && ((uintptr_t)p.out % 16 == 0);
  int ch = PC_RT;
  if (p.pro.n == 0) ch = PC_NONE;
  else if (p.pro.n == 1 && p.pro.op[0] == OP_LOG) ch = PC_LOG;
  CUtensorMap map;
  if (vec && make_pair_tensor_map(p, &map)) {  // rows on 16-byte boundaries: tensor copies into a stage ring
    if (p.epi.n) {
      if (ch == PC_LOG) return tma_launch<PC_LOG, true>(p, map, s);
      if (ch == PC_NONE) return tma_launch<PC_NONE, true>(p, map, s);
      return tma_launch<PC_RT, true>(p, map, s);
    }
    if (ch == PC_LOG) return tma_launch<PC_LOG, false>(p, map, s);
    if (ch == PC_NONE) return tma_launch<PC_NONE, false>(p, map, s);
    return tma_launch<PC_RT, false>(p, map, s);
  }
  if (ch == PC_LOG) return vec ? pair_launch<PC_LOG, true>(p, s) : pair_launch<PC_LOG, false>(p, s);
  if (ch == PC_NONE) return vec ? pair_launch<PC_NONE, true>(p, s) : pair_launch<PC_NONE, false>(p, s);
  return vec ? pair_launch<PC_RT, true>(p, s) : pair_launch<PC_RT, false>(p, s);
}

}  // namespace hlo
