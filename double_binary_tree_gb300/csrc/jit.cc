// Tree AllReduce kernels specialised at run time for the call's trees.
//
// The tree kernels of kernels.cuh and staged.cuh interpret a fold program per
// unit ([Course13] "每种 rank 的操作": a rank folds its input with its
// children's partials, post-order): one control byte per rank says how many
// partials to pop-fold and whether the rank's unit starts a new partial, and
// the partials live in register slots behind a warp-uniform switch.  That
// control flow costs issue slots on every unit.  Here the programs of one
// call become straight-line CUDA -- named partials, the pops and pushes fixed
// at compile time -- compiled with NVRTC together with the same kernel
// templates (kernels.cuh, staged.cuh under VR_JIT_TREE) and loaded as a
// library.  The generated steps are the program's steps, operand for
// operand, so the results are the interpreter's bit for bit.
//
// NVRTC is opened with dlopen: without it (or with VR_JIT=0) the built-in
// interpreting kernels run.  Kernels are cached per (architecture, element
// type, op, programs); the first call with new trees pays the compilation
// (a few seconds), each kernel kind separately when first needed.
#include <cuda_runtime.h>
#include <dlfcn.h>
#include <nvrtc.h>

#include <array>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "host.h"

namespace vr {
namespace {

// ------------------------------------------------------------------ NVRTC
struct Nvrtc {
  bool ok = false;
  std::string includeDir;  // CUDA headers (cuda_fp16.h, cuda_bf16.h)
  decltype(&nvrtcCreateProgram) create = nullptr;
  decltype(&nvrtcDestroyProgram) destroy = nullptr;
  decltype(&nvrtcAddNameExpression) addName = nullptr;
  decltype(&nvrtcCompileProgram) compile = nullptr;
  decltype(&nvrtcGetProgramLogSize) logSize = nullptr;
  decltype(&nvrtcGetProgramLog) log = nullptr;
  decltype(&nvrtcGetCUBINSize) cubinSize = nullptr;
  decltype(&nvrtcGetCUBIN) cubin = nullptr;
  decltype(&nvrtcGetLoweredName) lowered = nullptr;
};

std::string dir_of(const std::string& path) {
  const size_t k = path.find_last_of('/');
  return k == std::string::npos ? std::string(".") : path.substr(0, k);
}

bool file_exists(const std::string& p) {
  FILE* f = std::fopen(p.c_str(), "rb");
  if (!f) return false;
  std::fclose(f);
  return true;
}

// The CUDA root: CUDA_HOME / CUDA_PATH, the directory above the NVRTC that
// was opened, or /usr/local/cuda -- the first one holding cuda_fp16.h.
std::string cuda_include_dir(void* anySymbol) {
  std::vector<std::string> roots;
  for (const char* env : {"CUDA_HOME", "CUDA_PATH"})
    if (const char* v = std::getenv(env)) roots.push_back(v);
  Dl_info info;
  if (anySymbol && dladdr(anySymbol, &info) && info.dli_fname)
    roots.push_back(dir_of(dir_of(info.dli_fname)));
  roots.push_back("/usr/local/cuda");
  for (const std::string& r : roots)
    if (file_exists(r + "/include/cuda_fp16.h")) return r + "/include";
  return std::string();
}

const Nvrtc& nvrtc() {
  static const Nvrtc lib = [] {
    Nvrtc n;
    void* h = nullptr;
    std::vector<std::string> names = {"libnvrtc.so.13", "libnvrtc.so"};
    for (const char* env : {"CUDA_HOME", "CUDA_PATH"})
      if (const char* v = std::getenv(env)) names.push_back(std::string(v) + "/lib64/libnvrtc.so");
    names.push_back("/usr/local/cuda/lib64/libnvrtc.so");
    for (const std::string& name : names)
      if ((h = dlopen(name.c_str(), RTLD_NOW | RTLD_LOCAL))) break;
    if (!h) return n;
#define VR_SYM(field, name) n.field = reinterpret_cast<decltype(n.field)>(dlsym(h, #name))
    VR_SYM(create, nvrtcCreateProgram);
    VR_SYM(destroy, nvrtcDestroyProgram);
    VR_SYM(addName, nvrtcAddNameExpression);
    VR_SYM(compile, nvrtcCompileProgram);
    VR_SYM(logSize, nvrtcGetProgramLogSize);
    VR_SYM(log, nvrtcGetProgramLog);
    VR_SYM(cubinSize, nvrtcGetCUBINSize);
    VR_SYM(cubin, nvrtcGetCUBIN);
    VR_SYM(lowered, nvrtcGetLoweredName);
#undef VR_SYM
    n.includeDir = cuda_include_dir(reinterpret_cast<void*>(n.compile));
    n.ok = n.create && n.destroy && n.addName && n.compile && n.logSize && n.log &&
           n.cubinSize && n.cubin && n.lowered && !n.includeDir.empty();
    return n;
  }();
  return lib;
}

// The directory of the kernel sources: csrc/ beside this library (looked up
// once).
const std::string& source_dir() {
  static const std::string dir = [] {
    Dl_info info;
    if (!dladdr(reinterpret_cast<void*>(&source_dir), &info) || !info.dli_fname)
      return std::string();
    const std::string d = dir_of(info.dli_fname) + "/csrc";
    return file_exists(d + "/kernels.cuh") ? d : std::string();
  }();
  return dir;
}

// ------------------------------------------------------------- generation
const char* type_name(int dtype) {
  switch (dtype) {
    case VR_FLOAT32: return "float";
    case VR_FLOAT16: return "__half";
    case VR_BFLOAT16: return "__nv_bfloat16";
    default: return nullptr;
  }
}

// One program as straight-line steps on named partials s0..s{depth-1}:
// s{sp-1} is the top.  A pop folds the top into the partial beneath it
// (below op top), an add folds a rank's unit into the top (top op unit), a
// push starts a new partial -- the interpreter's operations in its order.
bool emit_program(const FoldProg& p, std::string* out) {
  char buf[96];
  int sp = 0;
  for (int k = 0; k < p.n; ++k) {
    const int c = p.ctl[k];
    for (int q = c & 15; q > 0; --q) {
      if (sp < 2) return false;
      --sp;
      std::snprintf(buf, sizeof buf, "  VR_J_POP(%d, %d)\n", sp - 1, sp);
      *out += buf;
    }
    if (c & 16) {
      if (sp >= kMaxStack) return false;
      std::snprintf(buf, sizeof buf, "  VR_J_PUSH(%d, %d)\n", sp, (int)p.rank[k]);
      ++sp;
    } else {
      if (sp < 1) return false;
      std::snprintf(buf, sizeof buf, "  VR_J_ADD(%d, %d)\n", sp - 1, (int)p.rank[k]);
    }
    *out += buf;
  }
  for (int q = p.tail; q > 0; --q) {
    if (sp < 2) return false;
    --sp;
    std::snprintf(buf, sizeof buf, "  VR_J_POP(%d, %d)\n", sp - 1, sp);
    *out += buf;
  }
  if (sp != 1) return false;
  *out += "  return Ln::encode(s0);\n";
  return true;
}

bool generate(const FoldProg* progs, int nProgs, std::string* src) {
  int depth = 1;
  for (int i = 0; i < nProgs; ++i) depth = progs[i].depth > depth ? progs[i].depth : depth;
  std::string s =
      "#define VR_JIT_TREE 1\n"
      "#include \"kernels.cuh\"\n"
      "#include \"staged.cuh\"\n"
      "namespace vr {\n"
      "#define VR_J_PUSH(d, r) Ln::decode(load_unit<T, NV>(src, r), s##d);\n"
      "#define VR_J_ADD(d, r) { typename Ln::L x_[Ln::N]; "
      "Ln::decode(load_unit<T, NV>(src, r), x_); "
      "_Pragma(\"unroll\") for (int e_ = 0; e_ < Ln::N; ++e_) s##d[e_] = Ln::op(s##d[e_], x_[e_]); }\n"
      "#define VR_J_POP(d, u) { "
      "_Pragma(\"unroll\") for (int e_ = 0; e_ < Ln::N; ++e_) s##d[e_] = Ln::op(s##d[e_], s##u[e_]); }\n"
      "template <typename T, int OP, int NV, class Src>\n"
      "__device__ __forceinline__ typename Unit<T, NV>::Raw jit_tree_fold(const Src& src, int t) {\n"
      "  typedef Lanes<T, OP, NV> Ln;\n";
  for (int d = 0; d < depth; ++d) s += "  typename Ln::L s" + std::to_string(d) + "[Ln::N];\n";
  s += "  switch (t) {\n";
  for (int i = 0; i < nProgs; ++i) {
    s += i == 0 ? "  default:\n  case 0: {\n" : "  case " + std::to_string(i) + ": {\n";
    if (!emit_program(progs[i], &s)) return false;
    s += "  }\n";
  }
  s += "  }\n}\n}  // namespace vr\n";
  *src = s;
  return true;
}

// The ring fold of one rank count R: the R units loaded in rank order
// (static ranks: the pointer table is read once, not per load), then block
// j's rotation j, j+1, ..., j-1 folded left to right from them -- the
// interpreter's folds, one straight-line case per j.
bool generate_ring(int R, std::string* src) {
  if (R < 1 || R > kMaxRanks) return false;
  std::string s =
      "#define VR_JIT_RING 1\n"
      "#include \"kernels.cuh\"\n"
      "#include \"staged.cuh\"\n"
      "namespace vr {\n"
      "#define VR_J_FOLD(v) { typename Ln::L x_[Ln::N]; Ln::decode(v, x_); "
      "_Pragma(\"unroll\") for (int e_ = 0; e_ < Ln::N; ++e_) acc[e_] = Ln::op(acc[e_], x_[e_]); }\n"
      "template <typename T, int OP, int NV, class Src>\n"
      "__device__ __forceinline__ typename Unit<T, NV>::Raw jit_ring_fold(const Src& src, int j) {\n"
      "  typedef Lanes<T, OP, NV> Ln;\n";
  for (int r = 0; r < R; ++r)
    s += "  const typename Unit<T, NV>::Raw v" + std::to_string(r) + " = load_unit<T, NV>(src, " +
         std::to_string(r) + ");\n";
  s += "  typename Ln::L acc[Ln::N];\n  switch (j) {\n";
  for (int j = 0; j < R; ++j) {
    s += j == 0 ? "  default:\n  case 0:\n" : "  case " + std::to_string(j) + ":\n";
    s += "    Ln::decode(v" + std::to_string(j) + ", acc);\n";
    for (int k = 1; k < R; ++k) s += "    VR_J_FOLD(v" + std::to_string((j + k) % R) + ")\n";
    s += "    break;\n";
  }
  s += "  }\n  return Ln::encode(acc);\n}\n}  // namespace vr\n";
  *src = s;
  return true;
}

// ------------------------------------------------------------------ cache
struct Entry {
  bool ok = false;
  cudaLibrary_t lib = nullptr;
  cudaKernel_t kernel = nullptr;
};
std::mutex g_jitMu;
std::map<std::string, Entry> g_cache;
long long g_compiled = 0, g_failed = 0;

std::string cache_key(int arch, int dtype, int op, int stack, bool small, const FoldProg* progs,
                      int nProgs) {
  std::string k = std::to_string(arch) + "/" + std::to_string(dtype) + "/" + std::to_string(op) +
                  "/" + std::to_string(stack) + "/" + (small ? "s/" : "g/");
  for (int i = 0; i < nProgs; ++i)
    k.append(reinterpret_cast<const char*>(&progs[i]), sizeof(FoldProg));
  return k;
}

// Compiles the register-path and staged tree kernels of `progs` for sm_<arch>a
// into a CUBIN.  Returns the lowered names in `names`.
// mode: kTreeAllReduce (progs, nProgs, stack) or kRingAllReduce (R).
// kind: 0 register path, 1 staged, 2 staged drawing its tiles (trees).
bool compile(int arch, int dtype, int op, int mode, int stack, bool small, int kind,
             const FoldProg* progs, int nProgs, int R, int minBlocks, std::string* cubin,
             std::string* name, std::string* log) {
  const Nvrtc& n = nvrtc();
  const std::string dir = source_dir();
  const char* T = type_name(dtype);
  if (!n.ok || dir.empty() || !T || (op != VR_SUM && op != VR_MAX)) return false;
  std::string src;
  if (mode == kTreeAllReduce ? !generate(progs, nProgs, &src) : !generate_ring(R, &src))
    return false;
  if (minBlocks > 0) src = "#define VR_JIT_MIN_BLOCKS " + std::to_string(minBlocks) + "\n" + src;
#ifdef VR_DEBUG_BOUNDS
  src = "#define VR_DEBUG_BOUNDS 1\n" + src;  // the bounds-checked build's kernels check too
#endif
  const int S = stack <= 4 ? 4 : 8;
  const std::string M = std::to_string(mode);
  const std::string expr =
      kind == 0 ? std::string("vr::allreduce_kernel<") + T + ", " + std::to_string(op) + ", " +
                      M + ", true, " + std::to_string(S) + (small ? ", true>" : ", false>")
                : std::string("vr::staged_kernel<") + T + ", " + std::to_string(op) + ", " + M +
                      ", " + std::to_string(S) + (kind == 2 ? ", true>" : ">");
  nvrtcProgram prog;
  if (n.create(&prog, src.c_str(), "vr_jit_tree.cu", 0, nullptr, nullptr) != NVRTC_SUCCESS)
    return false;
  n.addName(prog, expr.c_str());
  const std::string archOpt = "--gpu-architecture=sm_" + std::to_string(arch) + "a";
  const std::string inc1 = "--include-path=" + dir;
  const std::string inc2 = "--include-path=" + n.includeDir;
  const char* opts[] = {archOpt.c_str(), "-std=c++17", inc1.c_str(), inc2.c_str(),
                        "-default-device", "-lineinfo"};
  const nvrtcResult r = n.compile(prog, 6, opts);
  size_t ls = 0;
  if (n.logSize(prog, &ls) == NVRTC_SUCCESS && ls > 1 && log) {
    log->resize(ls);
    n.log(prog, &(*log)[0]);
  }
  bool ok = r == NVRTC_SUCCESS;
  size_t cs = 0;
  if (ok) ok = n.cubinSize(prog, &cs) == NVRTC_SUCCESS && cs > 0;
  if (ok) {
    cubin->resize(cs);
    ok = n.cubin(prog, &(*cubin)[0]) == NVRTC_SUCCESS;
  }
  if (ok) {
    const char* low = nullptr;
    ok = n.lowered(prog, expr.c_str(), &low) == NVRTC_SUCCESS && low;
    if (ok) *name = low;
  }
  n.destroy(&prog);
  return ok;
}

}  // namespace

bool jit_enabled() {
  if (option(kOptJit) == 0) return false;  // the option VR_JIT=0 turns the specialisation off
  return nvrtc().ok && !source_dir().empty();
}

namespace {

// The compiled kernel for `key`, compiling and loading it on first use.
vr_result_t cached_kernel(const std::string& key, int dtype, int op, int mode, int stack,
                          bool small, int kind, const FoldProg* progs, int nProgs, int R,
                          int minBlocks, int arch, const void** out) {
  std::lock_guard<std::mutex> g(g_jitMu);
  auto it = g_cache.find(key);
  if (it == g_cache.end()) {
    Entry e;
    std::string cubin, name;
    if (compile(arch, dtype, op, mode, stack, small, kind, progs, nProgs, R, minBlocks,
                &cubin, &name, nullptr) &&
        cudaLibraryLoadData(&e.lib, cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0) ==
            cudaSuccess)
      e.ok = cudaLibraryGetKernel(&e.kernel, e.lib, name.c_str()) == cudaSuccess;
    cudaGetLastError();  // a failed load leaves no sticky error; clear the last one
    ++(e.ok ? g_compiled : g_failed);
    it = g_cache.emplace(key, e).first;
  }
  if (!it->second.ok) return VR_ERR_UNSUPPORTED;
  *out = reinterpret_cast<const void*>(it->second.kernel);
  return VR_SUCCESS;
}

vr_result_t device_arch(int* arch) {
  int device = 0, major = 0, minor = 0;
  if (cudaGetDevice(&device) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return VR_ERR_CUDA;
  *arch = major * 10 + minor;
  return VR_SUCCESS;
}

}  // namespace

vr_result_t jit_tree_kernel(int dtype, int op, int stack, bool small, bool staged,
                            const FoldProg* progs, int nProgs, const void** out, int minBlocks,
                            bool drawn) {
  int arch = 0;
  const vr_result_t e = device_arch(&arch);
  if (e != VR_SUCCESS) return e;
  small = small && !staged;
  if (staged) minBlocks = 0;
  const int kind = staged ? (drawn ? 2 : 1) : 0;
  const std::string key = "t" + std::to_string(kind) + "/" + std::to_string(minBlocks) + "/" +
                          cache_key(arch, dtype, op, stack, small, progs, nProgs);
  return cached_kernel(key, dtype, op, kTreeAllReduce, stack, small, kind, progs, nProgs, 0,
                       minBlocks, arch, out);
}

vr_result_t jit_ring_kernel(int dtype, int op, int R, bool small, bool staged,
                            const void** out, int minBlocks) {
  int arch = 0;
  const vr_result_t e = device_arch(&arch);
  if (e != VR_SUCCESS) return e;
  small = small && !staged;
  if (staged) minBlocks = 0;
  const std::string key = std::string(staged ? "r1/" : "r0/") + std::to_string(minBlocks) + "/" +
                          std::to_string(arch) + "/" + std::to_string(dtype) + "/" +
                          std::to_string(op) + "/" + std::to_string(R) + (small ? "/s" : "/g");
  return cached_kernel(key, dtype, op, kRingAllReduce, 0, small, staged ? 1 : 0, nullptr, 0, R,
                       minBlocks, arch, out);
}

void jit_counts(long long* compiled, long long* failed) {
  std::lock_guard<std::mutex> g(g_jitMu);
  *compiled = g_compiled;
  *failed = g_failed;
}

// Compile-only check of the double binary tree of (nNodes, localRanks), all
// three kernel kinds: no device is touched.  The compiler's log goes to
// `log` (truncated).
vr_result_t jit_compile_dtree(int nNodes, int L, int dtype, int op, int arch,
                              size_t* cubinBytes, char* log, size_t logBytes) {
  FoldProg p[2];
  vr_result_t e = dtree_programs(nNodes, L, p);
  if (e != VR_SUCCESS) return e;
  const int stack = p[0].depth > p[1].depth ? p[0].depth : p[1].depth;
  if (!nvrtc().ok || source_dir().empty()) return VR_ERR_UNSUPPORTED;
  std::string text;
  *cubinBytes = 0;
  for (int kind = 0; kind < 3; ++kind) {
    std::string cubin, name;
    const bool ok = compile(arch, dtype, op, kTreeAllReduce, stack, false, kind, p, 2, 0, 0,
                            &cubin, &name, &text);
    if (log && logBytes) {
      std::strncpy(log, text.c_str(), logBytes - 1);
      log[logBytes - 1] = 0;
    }
    if (!ok) return VR_ERR_INTERNAL;
    *cubinBytes += cubin.size();
  }
  return VR_SUCCESS;
}

// Compile-only check of the ring fold of R ranks (both kernel kinds).
vr_result_t jit_compile_ring(int R, int dtype, int op, int arch, size_t* cubinBytes, char* log,
                             size_t logBytes) {
  if (R < 1 || R > kMaxRanks) return VR_ERR_INVALID_ARGUMENT;
  if (!nvrtc().ok || source_dir().empty()) return VR_ERR_UNSUPPORTED;
  std::string text;
  *cubinBytes = 0;
  for (int kind = 0; kind < 2; ++kind) {
    std::string cubin, name;
    if (!compile(arch, dtype, op, kRingAllReduce, 0, false, kind, nullptr, 0, R, 0, &cubin, &name,
                 &text)) {
      if (log && logBytes) {
        std::strncpy(log, text.c_str(), logBytes - 1);
        log[logBytes - 1] = 0;
      }
      return VR_ERR_INTERNAL;
    }
    *cubinBytes += cubin.size();
  }
  return VR_SUCCESS;
}

}  // namespace vr
