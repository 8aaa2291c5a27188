// Run-time generated kernels for 16-bit elementwise chains ("XLA:GPU Emitters", section "Loop emitter":
// the emitter produces one kernel per fusion, its ops written out as straight-line code over a linear
// walk of the output, with vectorized loads and stores).
//
// The interpreter kernels in k_elementwise.cu walk the chain's op list at run time; for a long chain on
// 16-bit values that walk costs as much as the arithmetic. Here the library writes the chain as CUDA C
// source (packed bf16x2 / f16x2 instructions in op order, bf16 tanh from the correctly rounded table),
// compiles it with NVRTC for this device's architecture and loads it through the driver API, once per
// (device, element type, op list); later calls reuse the kernel. Every op is the same instruction the
// interpreter issues, so the results are the same bits.
//
// NVRTC is opened with dlopen the first time a chain qualifies; when it cannot be opened, or a chain
// fails to compile, the interpreter kernels serve the call instead (hlo_jit_kernels reports -1 or the
// number of kernels built).
#include <cuda.h>
#include <cuda_fp16.h>
#include <dlfcn.h>
#include <nvrtc.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "async_copy.cuh"
#include "hlo_internal.h"

namespace hlo {
namespace {

// ---- NVRTC (dlopen) and the driver calls (runtime entry points) ---------------------------------------
struct NvrtcApi {
  bool ok = false;
  decltype(&nvrtcCreateProgram) create = nullptr;
  decltype(&nvrtcCompileProgram) compile = nullptr;
  decltype(&nvrtcGetCUBINSize) cubin_size = nullptr;
  decltype(&nvrtcGetCUBIN) cubin = nullptr;
  decltype(&nvrtcDestroyProgram) destroy = nullptr;
};

const NvrtcApi& nvrtc() {
  static NvrtcApi api = [] {
    NvrtcApi a;
    void* h = nullptr;
    for (const char* name : {"libnvrtc.so.13", "libnvrtc.so"}) {
      h = dlopen(name, RTLD_NOW | RTLD_LOCAL);
      if (h) break;
    }
    if (!h) {  // the toolkit's own directory, when it is not on the loader path
      const char* home = std::getenv("CUDA_HOME");
      const std::string dir = std::string(home && *home ? home : "/usr/local/cuda") + "/lib64/libnvrtc.so";
      h = dlopen(dir.c_str(), RTLD_NOW | RTLD_LOCAL);
    }
    if (!h) return a;
    a.create = reinterpret_cast<decltype(a.create)>(dlsym(h, "nvrtcCreateProgram"));
    a.compile = reinterpret_cast<decltype(a.compile)>(dlsym(h, "nvrtcCompileProgram"));
    a.cubin_size = reinterpret_cast<decltype(a.cubin_size)>(dlsym(h, "nvrtcGetCUBINSize"));
    a.cubin = reinterpret_cast<decltype(a.cubin)>(dlsym(h, "nvrtcGetCUBIN"));
    a.destroy = reinterpret_cast<decltype(a.destroy)>(dlsym(h, "nvrtcDestroyProgram"));
    a.ok = a.create && a.compile && a.cubin_size && a.cubin && a.destroy;
    return a;
  }();
  return api;
}

struct DriverApi {
  bool ok = false;
  CUresult (*load)(CUmodule*, const void*) = nullptr;
  CUresult (*get)(CUfunction*, CUmodule, const char*) = nullptr;
  CUresult (*set_attr)(CUfunction, CUfunction_attribute, int) = nullptr;
  CUresult (*occupancy)(int*, CUfunction, int, size_t) = nullptr;
  CUresult (*launch)(CUfunction, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned, CUstream,
                     void**, void**) = nullptr;
};

template <typename F>
bool entry(const char* name, F& fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  const cudaError_t pending = cudaPeekAtLastError();
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess) {
    fn = reinterpret_cast<F>(p);
    return true;
  }
  if (pending == cudaSuccess) cudaGetLastError();  // the lookup's own error
  return false;
}

const DriverApi& driver() {
  static DriverApi api = [] {
    DriverApi a;
    a.ok = entry("cuModuleLoadData", a.load) && entry("cuModuleGetFunction", a.get) &&
           entry("cuFuncSetAttribute", a.set_attr) && entry("cuOccupancyMaxActiveBlocksPerMultiprocessor", a.occupancy) &&
           entry("cuLaunchKernel", a.launch);
    return a;
  }();
  return api;
}

// The device address of this unit's fault word (the generated kernels record copy timeouts there; the
// word is read with the library's others by hlo_device_faults), once per device.
unsigned int* fault_word_address() {
  static std::mutex mu;
  static std::map<int, unsigned int*> addr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) return it->second;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_tu_faults) != cudaSuccess) {
    cudaGetLastError();
    p = nullptr;
  }
  addr[dev] = static_cast<unsigned int*>(p);
  return addr[dev];
}

// ---- source generation ---------------------------------------------------------------------------------
constexpr int kJitVecs = 2;                    // 16-byte vectors per thread and chunk
constexpr int kJitThreads = 1024 / kJitVecs;

// The packed constant of an op: the element type's bits of the value in both halves.
uint32_t splat_bits(float v, int dt) {
  uint32_t b;
  if (dt == BF16) {
    uint32_t f;
    std::memcpy(&f, &v, 4);
    b = f >> 16;  // the value is a bf16 value already: the low half is zero
  } else {
    const __half h = __float2half_rn(v);
    uint16_t u;
    std::memcpy(&u, &h, 2);
    b = u;
  }
  return b | (b << 16);
}

bool has_tanh(const Chain& c) {
  for (int k = 0; k < c.n; ++k)
    if (c.op[k] == OP_TANH) return true;
  return false;
}

bool reads_input(int op) { return op == OP_MUL_IN || op == OP_ADD_IN; }

// Where the generated kernel gets a chain's tanh from. Every op of a run that does not read the input
// x (constant adds and multiplies, negate, abs, tanh) is a function of the running 16-bit value alone,
// so a whole such run is one 65536-entry table: the run's ops applied to every bit pattern with the
// same instructions, once per chain, then one lookup per element instead of the run. The generator
// does that for a bf16 chain whose tanh ops all sit in one such run of two or more ops (GELU's
// multiply, tanh, add 1, multiply by 1/2); other chains with a tanh read the tanh table (64 KiB, indexed
// by |x|).
struct TablePlan {
  int kind = 0;            // 0: no table, 1: the tanh table, 2: a table of the run [run0, run1)
  int run0 = 0, run1 = 0;
  int bytes() const { return kind == 0 ? 0 : kind == 1 ? 65536 : 131072; }
};

TablePlan plan_table(const Chain& c, int dt) {
  TablePlan p;
  if (!has_tanh(c)) return p;
  p.kind = 1;
  int runs_with_tanh = 0, r0 = 0, r1 = 0;
  for (int k = 0; k < c.n;) {
    if (reads_input(c.op[k])) {
      ++k;
      continue;
    }
    int e = k, nt = 0;
    for (; e < c.n && !reads_input(c.op[e]); ++e) nt += c.op[e] == OP_TANH;
    if (nt) {
      ++runs_with_tanh;
      r0 = k;
      r1 = e;
    }
    k = e;
  }
  if (dt == BF16 && runs_with_tanh == 1 && r1 - r0 >= 2) {
    p.kind = 2;
    p.run0 = r0;
    p.run1 = r1;
  }
  return p;
}

// The ops [k0, k1) of the chain as straight-line code on the packed pair v (x: the input pair, t: the
// table).
std::string chain_body(const Chain& c, int dt, int k0, int k1) {
  std::string s;
  char line[128];
  for (int k = k0; k < k1; ++k) {
    switch (c.op[k]) {
      case OP_MUL_IN: s += "  v = hmul(v, x);\n"; break;
      case OP_ADD_IN: s += "  v = hadd(v, x);\n"; break;
      case OP_MUL_CONST:
        std::snprintf(line, sizeof line, "  v = hmul(v, 0x%08Xu);\n", splat_bits(c.imm[k], dt));
        s += line;
        break;
      case OP_ADD_CONST:
        std::snprintf(line, sizeof line, "  v = hadd(v, 0x%08Xu);\n", splat_bits(c.imm[k], dt));
        s += line;
        break;
      case OP_NEG: s += "  v ^= 0x80008000u;\n"; break;
      case OP_ABS: s += "  v &= 0x7FFF7FFFu;\n"; break;
      case OP_TANH: s += "  v = htanh(v, t);\n"; break;
      default: return std::string();  // not generated
    }
  }
  return s;
}

// The generated kernel streams the array through shared memory in 16 KiB chunks of 1024 vectors. Block b
// of G takes chunks b, b + G, b + 2G, ... of the whole rounds of G chunks, then an even share of what is
// left (the remainder's vectors split G ways, so no block streams a whole extra chunk). One block per
// SM keeps a ring of chunks in flight as 1-D bulk copies completing on mbarriers, issued up front by
// thread 0 (with the chain's table, if any: the 64 KiB tanh table or a 128 KiB run table) and refilled
// by the last warp to finish with a chunk, so an SM asks for its first 96-192 KiB of input at launch
// rather than a few vectors per thread at a time. Each thread takes kJitVecs vectors of a chunk,
// applies the chain and stores them straight to global memory; the last n % 8 elements are read
// directly by the last block. Every wait is bounded: on a timeout the block records the fault in the
// library's fault word, waits (bounded) for the copies it still has in flight and returns.
constexpr int kChunkVecs = 1024;
constexpr int kChunkBytes = kChunkVecs * 16;

int ring_stages(int table_bytes) {
  const int room = 227 * 1024 - table_bytes - 512;  // barriers and counters in the last 512 B
  const int ns = room / kChunkBytes;
  return ns < 12 ? ns : 12;
}

size_t ring_smem(int table_bytes) { return (size_t)table_bytes + (size_t)ring_stages(table_bytes) * kChunkBytes + 512; }

std::string kernel_source(const Chain& c, int dt, const TablePlan& tp) {
  const char* ty = dt == BF16 ? "bf16" : "f16";
  const bool tanh = tp.kind != 0;  // a table in shared memory
  std::string src;
  src += "#define NS " + std::to_string(ring_stages(tp.bytes())) + "\n";
  src += "#define TB " + std::to_string(tp.bytes()) + "\n";
  src += "#define CB " + std::to_string(kChunkBytes) + "\n";
  src += "typedef unsigned int u32;\n";
  src += "struct alignas(16) v4 { u32 a, b, c, d; };\n";
  src += std::string("__device__ __forceinline__ u32 hadd(u32 a, u32 b) { u32 r; asm(\"add.rn.") + ty +
         "x2 %0, %1, %2;\" : \"=r\"(r) : \"r\"(a), \"r\"(b)); return r; }\n";
  src += std::string("__device__ __forceinline__ u32 hmul(u32 a, u32 b) { u32 r; asm(\"mul.rn.") + ty +
         "x2 %0, %1, %2;\" : \"=r\"(r) : \"r\"(a), \"r\"(b)); return r; }\n";
  src +=
      "__device__ __forceinline__ u32 prmt(u32 a, u32 b, u32 s) { u32 r; asm(\"prmt.b32 %0, %1, %2, %3;\" : \"=r\"(r) : "
      "\"r\"(a), \"r\"(b), \"r\"(s)); return r; }\n"
      // tanh of a bf16 pair: the table entry of |x| with the sign of x
      "__device__ __forceinline__ u32 htanh(u32 w, const unsigned short* t) {\n"
      "  const u32 a = w & 0x7FFF7FFFu;\n"
      "  return prmt((u32)t[a & 0xFFFFu], (u32)t[a >> 16], 0x5410u) | (w & 0x80008000u);\n"
      "}\n"
      // a pair through the run's table (indexed by all 16 bits)
      "__device__ __forceinline__ u32 hlook(u32 w, const unsigned short* t) {\n"
      "  return prmt((u32)t[w & 0xFFFFu], (u32)t[w >> 16], 0x5410u);\n"
      "}\n"
      "__device__ __forceinline__ v4 ld4(const v4* p) { v4 r; asm volatile(\"ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\" "
      ": \"=r\"(r.a), \"=r\"(r.b), \"=r\"(r.c), \"=r\"(r.d) : \"l\"(p)); return r; }\n"
      "__device__ __forceinline__ void st4(v4* p, v4 v) { asm volatile(\"st.global.v4.u32 [%0], {%1, %2, %3, %4};\" :: "
      "\"l\"(p), \"r\"(v.a), \"r\"(v.b), \"r\"(v.c), \"r\"(v.d) : \"memory\"); }\n"
      "__device__ __forceinline__ v4 lds4(u32 a) { v4 r; asm volatile(\"ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\" "
      ": \"=r\"(r.a), \"=r\"(r.b), \"=r\"(r.c), \"=r\"(r.d) : \"r\"(a) : \"memory\"); return r; }\n"
      // mbarriers and 1-D bulk copies
      "__device__ __forceinline__ void bar_init(u32 b, u32 c) { asm volatile(\"mbarrier.init.shared::cta.b64 [%0], %1;\" "
      ":: \"r\"(b), \"r\"(c)); }\n"
      "__device__ __forceinline__ void expect(u32 b, u32 n) { asm volatile(\"mbarrier.arrive.expect_tx.shared::cta.b64 _, "
      "[%0], %1;\" :: \"r\"(b), \"r\"(n) : \"memory\"); }\n"
      "__device__ __forceinline__ void bulk(u32 d, const void* g, u32 n, u32 b) { asm volatile(\"cp.async.bulk.shared::"
      "cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\" :: \"r\"(d), \"l\"(g), \"r\"(n), \"r\"(b) : "
      "\"memory\"); }\n"
      // waits for phase `par`; false after about a second (2^31 cycles) without it
      "__device__ __forceinline__ bool bar_wait(u32 b, u32 par) {\n"
      "  long long t0 = -1;\n"
      "  while (true) {\n"
      "    u32 d;\n"
      "    asm volatile(\"{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }\" "
      ": \"=r\"(d) : \"r\"(b), \"r\"(par) : \"memory\");\n"
      "    if (d) return true;\n"
      "    const long long now = clock64();\n"
      "    if (t0 < 0) t0 = now; else if (now - t0 > 2000000000LL) return false;\n"
      "  }\n"
      "}\n";
  src += "__device__ __forceinline__ u32 f(u32 x, const unsigned short* t) {\n  u32 v = x;\n";
  if (tp.kind == 2) {
    src += chain_body(c, dt, 0, tp.run0);
    src += "  v = hlook(v, t);\n";
    src += chain_body(c, dt, tp.run1, c.n);
  } else {
    src += chain_body(c, dt, 0, c.n);
  }
  src += "  return v;\n}\n";
  if (tp.kind == 2)  // the run's table: every bit pattern through the run's ops (tg: the tanh table)
    src += "extern \"C\" __global__ void hlo_jit_table(const unsigned short* __restrict__ tg, unsigned short* __restrict__ dst) "
           "{\n"
           "  const u32 p = blockIdx.x * blockDim.x + threadIdx.x;\n"
           "  if (p >= 65536u) return;\n"
           "  const unsigned short* t = tg;\n"
           "  u32 v = p | (p << 16);\n" +
           chain_body(c, dt, tp.run0, tp.run1) +
           "  dst[p] = (unsigned short)(v & 0xFFFFu);\n"
           "}\n";
  src +=
      "__device__ __forceinline__ v4 f4(v4 w, const unsigned short* t) { return v4{f(w.a, t), f(w.b, t), f(w.c, t), f(w.d, t)}; "
      "}\n";
  src += "#define VPT " + std::to_string(kJitVecs) + "\n#define CV " + std::to_string(kChunkVecs) + "\n";
  src += "extern \"C\" __global__ void __launch_bounds__(" + std::to_string(kJitThreads) +
         ", 1) hlo_jit_chain(const v4* __restrict__ in, v4* __restrict__ out, long long n, const v4* __restrict__ tg, "
         "u32* __restrict__ fault) {\n"
         "  extern __shared__ __align__(128) unsigned char sm[];\n"
         "  const unsigned short* t = reinterpret_cast<const unsigned short*>(sm);\n"
         "  const u32 ring = (u32)__cvta_generic_to_shared(sm + TB);\n"
         "  const u32 bars = ring + NS * CB;\n"  // NS chunk barriers, then the table's
         "  int* done = reinterpret_cast<int*>(sm + TB + NS * CB + (NS + 1) * 8);\n"
         "  const long long nvec = n >> 3, G = gridDim.x, b = blockIdx.x;\n"
         // whole rounds of G chunks, then block b's share [l0, l0 + ln) of the remaining vectors
         "  const long long rounds = nvec / (G * CV), rest = nvec - rounds * G * CV;\n"
         "  const long long lq = rest / G, lr = rest % G;\n"
         "  const long long l0 = rounds * G * CV + b * lq + (b < lr ? b : lr), ln = lq + (b < lr ? 1 : 0);\n"
         "  const long long mine = rounds + (ln > 0 ? 1 : 0);\n"
         "  const int tid = threadIdx.x;\n"
         "  if (tid == 0) {\n"
         "    for (int s = 0; s < NS; ++s) { bar_init(bars + 8 * s, 1); done[s] = 0; }\n"
         "    bar_init(bars + 8 * NS, 1);\n"
         "    asm volatile(\"fence.mbarrier_init.release.cluster;\" ::: \"memory\");\n";
  if (tanh)
    src += "    expect(bars + 8 * NS, TB); bulk((u32)__cvta_generic_to_shared(sm), tg, TB, bars + 8 * NS);\n";
  src +=
      "    for (int s = 0; s < NS && s < mine; ++s) {\n"
      "      const long long c0 = s < rounds ? (b + s * G) * CV : l0, cn = s < rounds ? CV : ln;\n"
      "      expect(bars + 8 * s, (u32)cn * 16); bulk(ring + s * CB, in + c0, (u32)cn * 16, bars + 8 * s);\n"
      "    }\n"
      "  }\n"
      "  __syncthreads();\n";
  src += tanh ? "  bool ok = __all_sync(0xFFFFFFFFu, bar_wait(bars + 8 * NS, 0));\n" : "  bool ok = true;\n";
  src +=
      "  long long k = 0;\n"
      "  int s = 0;\n"
      "  u32 ph = 0;\n"
      "  for (; ok && k < mine; ++k) {\n"
      // the warp decides together (the __syncwarp below needs all of its lanes)
      "    if (!__all_sync(0xFFFFFFFFu, bar_wait(bars + 8 * s, ph))) { ok = false; break; }\n"
      "    const long long c0 = k < rounds ? (b + k * G) * CV : l0;\n"
      "    const int cn = k < rounds ? CV : (int)ln;\n"
      "    v4 x[VPT];\n"
      "#pragma unroll\n"
      "    for (int j = 0; j < VPT; ++j) if (tid + j * (CV / VPT) < cn) x[j] = lds4(ring + s * CB + (tid + j * (CV / VPT)) * 16);\n"
      "#pragma unroll\n"
      "    for (int j = 0; j < VPT; ++j) if (tid + j * (CV / VPT) < cn) st4(out + c0 + tid + j * (CV / VPT), f4(x[j], t));\n"
      // the warp's vectors are in registers (the stores above depend on them): the last warp refills
      "    __syncwarp();\n"
      "    if ((tid & 31) == 0) {\n"
      "      __threadfence_block();\n"
      "      if (atomicAdd(&done[s], 1) == (int)(blockDim.x / 32) - 1) {\n"
      "        done[s] = 0;\n"
      "        const long long nk = k + NS;\n"
      "        if (nk < mine) {\n"
      "          const long long d0 = nk < rounds ? (b + nk * G) * CV : l0, dn = nk < rounds ? CV : ln;\n"
      "          asm volatile(\"fence.proxy.async.shared::cta;\" ::: \"memory\");\n"
      "          expect(bars + 8 * s, (u32)dn * 16);\n"
      "          bulk(ring + s * CB, in + d0, (u32)dn * 16, bars + 8 * s);\n"
      "        }\n"
      "      }\n"
      "    }\n"
      "    if (++s == NS) { s = 0; ph ^= 1u; }\n"
      "  }\n"
      "  if (!ok) {\n"
      // a copy did not arrive in time: record it, wait (bounded) for the copies this block may still have
      // in flight (the table and chunks k .. k + NS - 1) and return
      "    if (tid == 0) atomicOr(fault, 1u);\n";
  if (tanh) src += "    bar_wait(bars + 8 * NS, 0);\n";
  src +=
      "    for (long long q2 = k; q2 < k + NS && q2 < mine; ++q2) bar_wait(bars + 8 * (int)(q2 % NS), (u32)((q2 / NS) & 1));\n"
      "    return;\n"
      "  }\n"
      "  if (b == G - 1) {\n"
      "    const unsigned short* i16 = reinterpret_cast<const unsigned short*>(in);\n"
      "    unsigned short* o16 = reinterpret_cast<unsigned short*>(out);\n"
      "    for (long long e = nvec * 8 + tid; e < n; e += blockDim.x) o16[e] = (unsigned short)(f((u32)i16[e], t) & 0xFFFFu);\n"
      "  }\n"
      "}\n";
  return src;
}

std::string chain_key(const Chain& c, int dt) {
  std::string k = dt == BF16 ? "bf16" : "f16";
  char buf[48];
  for (int i = 0; i < c.n; ++i) {
    std::snprintf(buf, sizeof buf, ":%d", c.op[i]);
    k += buf;
    if (c.op[i] == OP_MUL_CONST || c.op[i] == OP_ADD_CONST) {
      std::snprintf(buf, sizeof buf, "=%08X", splat_bits(c.imm[i], dt));
      k += buf;
    }
  }
  return k;
}

struct JitKernel {
  CUfunction fn = nullptr;  // null: the chain did not compile (the interpreter serves it)
  int blocks_per_sm = 0;
  size_t smem = 0;
  TablePlan tp;
  const void* table = nullptr;     // what the kernel copies into shared memory (tanh or run table)
  cudaEvent_t ready = nullptr;     // run table: recorded after it was built, on stream built_on
  cudaStream_t built_on = nullptr;
};

// Run tables, in this unit's device memory: a chain's table is built into a free slot the first time
// the chain runs on a device and stays there; chains past the last slot use the tanh table instead.
constexpr int kRunTableSlots = 8;
static __device__ __align__(16) uint16_t g_run_tables[kRunTableSlots][65536];

uint16_t* run_table_slot(int dev) {
  static std::map<int, int> used;  // callers hold g_mu
  int& k = used[dev];
  if (k >= kRunTableSlots) return nullptr;
  void* base = nullptr;
  if (cudaGetSymbolAddress(&base, g_run_tables) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<uint16_t*>(base) + (size_t)65536 * k++;
}

std::mutex g_mu;
std::map<std::pair<int, std::string>, JitKernel> g_cache;

// Compiles the chain for the current device (or returns the cached result); a run table is built on
// stream s. With build_new false only a cached kernel is returned (a default one, no kernel, otherwise).
JitKernel build(const Chain& c, int dt, int dev, cudaStream_t s, bool build_new) {
  const auto key = std::make_pair(dev, chain_key(c, dt));
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_cache.find(key);
  if (it != g_cache.end()) return it->second;
  if (!build_new) return JitKernel{};
  JitKernel jk;
  cudaSetDevice(dev);  // makes the device's primary context current for the driver calls below
  const NvrtcApi& nv = nvrtc();
  const DriverApi& dr = driver();
  int major = 0, minor = 0;
  const void* tg = has_tanh(c) ? tanh_table_address() : nullptr;
  TablePlan tp = plan_table(c, dt);
  uint16_t* slot = nullptr;
  if (tp.kind == 2 && !(slot = run_table_slot(dev))) tp = TablePlan{1, 0, 0};
  if (nv.ok && dr.ok && (tp.kind == 0 || tg) &&
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess) {
    const std::string src = kernel_source(c, dt, tp);
    nvrtcProgram prog = nullptr;
    if (nv.create(&prog, src.c_str(), "hlo_jit_chain.cu", 0, nullptr, nullptr) == NVRTC_SUCCESS) {
      const std::string arch = "--gpu-architecture=sm_" + std::to_string(major * 10 + minor) + (major >= 9 ? "a" : "");
      const char* opts[] = {arch.c_str(), "-std=c++17"};
      size_t size = 0;
      std::vector<char> cubin;
      if (nv.compile(prog, 2, opts) == NVRTC_SUCCESS && nv.cubin_size(prog, &size) == NVRTC_SUCCESS && size > 0) {
        cubin.resize(size);
        if (nv.cubin(prog, cubin.data()) != NVRTC_SUCCESS) cubin.clear();
      }
      nv.destroy(&prog);
      CUmodule mod = nullptr;
      CUfunction fn = nullptr, table_fn = nullptr;
      if (!cubin.empty() && dr.load(&mod, cubin.data()) == CUDA_SUCCESS &&
          dr.get(&fn, mod, "hlo_jit_chain") == CUDA_SUCCESS &&
          (tp.kind != 2 || dr.get(&table_fn, mod, "hlo_jit_table") == CUDA_SUCCESS)) {
        const size_t smem = ring_smem(tp.bytes());
        int nb = 0;
        bool ok = dr.set_attr(fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, (int)smem) == CUDA_SUCCESS &&
                  dr.occupancy(&nb, fn, kJitThreads, smem) == CUDA_SUCCESS && nb > 0;
        cudaEvent_t ready = nullptr;
        if (ok && tp.kind == 2) {  // build the run's table once, ordered before every use
          void* targs[] = {const_cast<void**>(&tg), &slot};
          ok = dr.launch(table_fn, 256, 1, 1, 256, 1, 1, 0, reinterpret_cast<CUstream>(s), targs, nullptr) == CUDA_SUCCESS &&
               cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) == cudaSuccess &&
               cudaEventRecord(ready, s) == cudaSuccess;
        }
        if (ok) {
          jk.fn = fn;
          jk.blocks_per_sm = nb;
          jk.smem = smem;
          jk.tp = tp;
          jk.table = tp.kind == 2 ? static_cast<const void*>(slot) : tg;
          jk.ready = ready;
          jk.built_on = s;
        }
      }
    }
  }
  g_cache[key] = jk;
  return jk;
}

}  // namespace

// The chains the generator writes: every op rounded to the 16-bit type, add / multiply by the input or
// a constant, negate, absolute value, and tanh on bf16 (from its table).
bool jit_chain_ok(const Chain& pro, const Chain& epi, int dt) {
  if ((dt != BF16 && dt != F16) || epi.n != 0 || !pro.round16 || pro.n == 0) return false;
  for (int k = 0; k < pro.n; ++k) {
    const int op = pro.op[k];
    if (op == OP_TANH && dt != BF16) return false;
    if (op != OP_MUL_IN && op != OP_ADD_IN && op != OP_MUL_CONST && op != OP_ADD_CONST && op != OP_NEG &&
        op != OP_ABS && op != OP_TANH)
      return false;
  }
  return true;
}

cudaError_t launch_jit_chain(const void* in, void* out, int64_t n, int dt, const Chain& pro, cudaStream_t s,
                             bool* used) {
  *used = false;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // While s is being captured into a graph, work enqueued on it is recorded, not run: a chain's first
  // use (which builds its run table on s) and a wait on the table's event both stay out of the capture,
  // so the interpreter takes the call unless the chain's kernel was built before and has no run table.
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &capture);
  if (e != cudaSuccess) return e;
  const bool capturing = capture != cudaStreamCaptureStatusNone;
  const JitKernel jk = build(pro, dt, dev, s, !capturing);
  if (!jk.fn || (capturing && jk.ready)) return cudaSuccess;  // the interpreter takes the call
  const void* tg = jk.table;
  if (jk.ready && s != jk.built_on) {  // the run table was built on another stream
    e = cudaStreamWaitEvent(s, jk.ready, 0);
    if (e != cudaSuccess) return e;
  }
  unsigned int* fault = fault_word_address();
  if (!fault) return cudaSuccess;
  // one block per SM; fewer for small arrays (at least 256 vectors, 4 KiB, per block)
  int64_t blocks = n / 8 / 256;
  const int64_t cap = (int64_t)device_sm_count() * jk.blocks_per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  long long nn = (long long)n;
  void* args[] = {const_cast<void**>(&in), &out, &nn, const_cast<void**>(&tg), &fault};
  const CUresult r = driver().launch(jk.fn, (unsigned)blocks, 1, 1, kJitThreads, 1, 1, (unsigned)jk.smem,
                                     reinterpret_cast<CUstream>(s), args, nullptr);
  if (r != CUDA_SUCCESS) return cudaErrorLaunchFailure;
  *used = true;
  return cudaSuccess;
}

bool jit_chain_source(const Chain& pro, int dt, std::string* out) {
  Chain none;
  std::memset(&none, 0, sizeof none);
  if (!jit_chain_ok(pro, none, dt)) return false;
  *out = kernel_source(pro, dt, plan_table(pro, dt));
  return true;
}

int jit_chain_kernels() {
  if (!nvrtc().ok || !driver().ok) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  int count = 0;
  for (const auto& kv : g_cache)
    if (kv.first.first == dev && kv.second.fn) ++count;
  return count;
}

}  // namespace hlo
