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

// ---- source generation ---------------------------------------------------------------------------------
constexpr int kJitThreads = 512;

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

std::string chain_body(const Chain& c, int dt) {
  std::string s;
  char line[128];
  for (int k = 0; k < c.n; ++k) {
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

std::string kernel_source(const Chain& c, int dt) {
  const char* ty = dt == BF16 ? "bf16" : "f16";
  std::string src;
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
      "__device__ __forceinline__ v4 ld4(const v4* p) { v4 r; asm volatile(\"ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\" "
      ": \"=r\"(r.a), \"=r\"(r.b), \"=r\"(r.c), \"=r\"(r.d) : \"l\"(p)); return r; }\n"
      "__device__ __forceinline__ void st4(v4* p, v4 v) { asm volatile(\"st.global.v4.u32 [%0], {%1, %2, %3, %4};\" :: "
      "\"l\"(p), \"r\"(v.a), \"r\"(v.b), \"r\"(v.c), \"r\"(v.d) : \"memory\"); }\n";
  src += "__device__ __forceinline__ u32 f(u32 x, const unsigned short* t) {\n  u32 v = x;\n";
  src += chain_body(c, dt);
  src += "  return v;\n}\n";
  src +=
      "__device__ __forceinline__ v4 f4(v4 w, const unsigned short* t) { return v4{f(w.a, t), f(w.b, t), f(w.c, t), f(w.d, t)}; "
      "}\n";
  src += "extern \"C\" __global__ void __launch_bounds__(" + std::to_string(kJitThreads) +
         ") hlo_jit_chain(const v4* __restrict__ in, v4* __restrict__ out, long long n, const v4* __restrict__ tg) {\n"
         "  extern __shared__ v4 tt4[];\n"
         "  const unsigned short* t = reinterpret_cast<const unsigned short*>(tt4);\n"
         "  const long long nvec = n >> 3, nth = (long long)gridDim.x * blockDim.x;\n"
         "  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;\n"
         "  const long long base = (gt >> 5) * 128 + (threadIdx.x & 31);\n"  // a warp's four loads: 512 B each
         "  const long long rounds = nvec / (4 * nth);\n"
         "  v4 x0, x1, x2, x3;\n"
         "  if (rounds > 0) { x0 = ld4(in + base); x1 = ld4(in + base + 32); x2 = ld4(in + base + 64); x3 = ld4(in + base + 96); }\n";
  if (has_tanh(c))
    src +=
        "  for (int i = threadIdx.x; i < 4096; i += blockDim.x) tt4[i] = ld4(tg + i);\n"
        "  __syncthreads();\n";
  src +=
      "  for (long long r = 0; r < rounds; ++r) {\n"
      "    const long long b = r * 4 * nth + base;\n"
      "    const v4 y0 = x0, y1 = x1, y2 = x2, y3 = x3;\n"
      "    if (r + 1 < rounds) { const long long c = b + 4 * nth; x0 = ld4(in + c); x1 = ld4(in + c + 32); x2 = ld4(in + c + 64); "
      "x3 = ld4(in + c + 96); }\n"
      "    st4(out + b, f4(y0, t)); st4(out + b + 32, f4(y1, t)); st4(out + b + 64, f4(y2, t)); st4(out + b + 96, f4(y3, t));\n"
      "  }\n"
      "  for (long long i = rounds * 4 * nth + gt; i < nvec; i += nth) st4(out + i, f4(ld4(in + i), t));\n"
      "  const unsigned short* i16 = reinterpret_cast<const unsigned short*>(in);\n"
      "  unsigned short* o16 = reinterpret_cast<unsigned short*>(out);\n"
      "  for (long long e = nvec * 8 + gt; e < n; e += nth) o16[e] = (unsigned short)(f((u32)i16[e], t) & 0xFFFFu);\n"
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
};

std::mutex g_mu;
std::map<std::pair<int, std::string>, JitKernel> g_cache;

// Compiles the chain for the current device (or returns the cached result).
JitKernel build(const Chain& c, int dt, int dev) {
  const auto key = std::make_pair(dev, chain_key(c, dt));
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_cache.find(key);
  if (it != g_cache.end()) return it->second;
  JitKernel jk;
  cudaSetDevice(dev);  // makes the device's primary context current for the driver calls below
  const NvrtcApi& nv = nvrtc();
  const DriverApi& dr = driver();
  int major = 0, minor = 0;
  if (nv.ok && dr.ok && cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess) {
    const std::string src = kernel_source(c, dt);
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
      CUfunction fn = nullptr;
      if (!cubin.empty() && dr.load(&mod, cubin.data()) == CUDA_SUCCESS &&
          dr.get(&fn, mod, "hlo_jit_chain") == CUDA_SUCCESS) {
        const size_t smem = has_tanh(c) ? 32768 * sizeof(uint16_t) : 0;
        int nb = 0;
        if (dr.set_attr(fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, (int)smem) == CUDA_SUCCESS &&
            dr.occupancy(&nb, fn, kJitThreads, smem) == CUDA_SUCCESS && nb > 0) {
          jk.fn = fn;
          jk.blocks_per_sm = nb;
          jk.smem = smem;
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
  const JitKernel jk = build(pro, dt, dev);
  if (!jk.fn) return cudaSuccess;  // the interpreter takes the call
  const void* tg = has_tanh(pro) ? tanh_table_address() : nullptr;
  if (has_tanh(pro) && !tg) return cudaSuccess;
  int64_t blocks = (n / 32 + kJitThreads - 1) / kJitThreads;
  const int64_t cap = (int64_t)device_sm_count() * jk.blocks_per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  long long nn = (long long)n;
  void* args[] = {const_cast<void**>(&in), &out, &nn, const_cast<void**>(&tg)};
  const CUresult r = driver().launch(jk.fn, (unsigned)blocks, 1, 1, kJitThreads, 1, 1, (unsigned)jk.smem,
                                     reinterpret_cast<CUstream>(s), args, nullptr);
  if (r != CUDA_SUCCESS) return cudaErrorLaunchFailure;
  *used = true;
  return cudaSuccess;
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
