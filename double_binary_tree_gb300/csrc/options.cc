// Tuning and test options: read from the environment once, at the first
// call that needs one, and changed afterwards only through vr_set_option.
// No option changes a result, only which kernel computes it (or what the
// library prints), so none is consulted on the device.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "host.h"

namespace vr {
namespace {

struct Spec {
  const char* name;
  long long dflt;  // -1: the call site's own default
};

// Index = Option.
const Spec kSpecs[kOptCount] = {
    {"VR_KERNEL_PATH", 0},        {"VR_JIT", 1},
    {"VR_JIT_RING", 2},           {"VR_JIT_OCC", 1},
    {"VR_SMALL_RANKS", 1},        {"VR_PDL", 1},
    {"VR_SPREAD", 1},             {"VR_STAGED_MIN_BYTES", 16ll << 20},
    {"VR_STAGED_TILE_BYTES", 0},  {"VR_STAGED_MIN_STAGES", -1},
    {"VR_STAGED_STAGES", 0},      {"VR_AG_TILE", -1},
    {"VR_AG_STAGES", -1},         {"VR_AG_CTAS", -1},
    {"VR_AG_ORDER", 0},           {"VR_SCHED", 1},
    {"VR_DEBUG", 0},
};

std::atomic<long long> g_values[kOptCount];
std::once_flag g_once;

// The environment's text of one option as a value: VR_KERNEL_PATH takes
// "register" (1) or "staged" (2), VR_DEBUG a comma-separated list of
// subsystems ("GRAPH" is bit 0), the others a decimal integer.
long long parse(int o, const char* v) {
  if (o == kOptKernelPath) {
    if (std::strcmp(v, "register") == 0) return 1;
    if (std::strcmp(v, "staged") == 0) return 2;
    return 0;
  }
  if (o == kOptDebug) {
    long long bits = 0;
    const char* p = v;
    while (*p) {
      const char* e = std::strchr(p, ',');
      const size_t n = e ? (size_t)(e - p) : std::strlen(p);
      if (n == 5 && std::strncmp(p, "GRAPH", 5) == 0) bits |= kDebugGraph;
      if (!e) break;
      p = e + 1;
    }
    return bits;
  }
  char* end = nullptr;
  const long long x = std::strtoll(v, &end, 10);
  return end != v && x >= 0 ? x : kSpecs[o].dflt;
}

void load_environment() {
  for (int o = 0; o < kOptCount; ++o) {
    const char* v = std::getenv(kSpecs[o].name);
    g_values[o].store(v ? parse(o, v) : kSpecs[o].dflt, std::memory_order_relaxed);
  }
}

int find(const char* name) {
  if (!name) return -1;
  for (int o = 0; o < kOptCount; ++o)
    if (std::strcmp(name, kSpecs[o].name) == 0) return o;
  return -1;
}

}  // namespace

long long option(Option o) {
  std::call_once(g_once, load_environment);
  return g_values[o].load(std::memory_order_relaxed);
}

long long option_or(Option o, long long dflt) {
  const long long v = option(o);
  return v < 0 ? dflt : v;
}

}  // namespace vr

using namespace vr;

extern "C" {

vr_result_t vr_set_option(const char* name, long long value) {
  const int o = find(name);
  if (o < 0 || value < -1) return VR_ERR_INVALID_ARGUMENT;
  std::call_once(g_once, load_environment);
  g_values[o].store(value == -1 ? kSpecs[o].dflt : value, std::memory_order_relaxed);
  return VR_SUCCESS;
}

vr_result_t vr_get_option(const char* name, long long* value) {
  const int o = find(name);
  if (o < 0 || !value) return VR_ERR_INVALID_ARGUMENT;
  *value = option((Option)o);
  return VR_SUCCESS;
}

}  // extern "C"
