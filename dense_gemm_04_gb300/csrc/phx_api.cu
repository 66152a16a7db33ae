// phx_api.cu -- the C ABI of libphx (include/phx.h): argument checks, per-device state,
// configuration choice, the autotuner, and the device status word.
//
// The operation and its argument list follow the kernel signature of "gemm, f32"
// (phobos-lang.dev/docs/examples/gemm-fp32/): gemm(A: tensor<f32>[M, K], B: tensor<f32>[K, N],
// C: tensor<f32>[M, N], alpha: f32, beta: f32).  The pages' launcher traps when the @aligned
// promise is broken ("The attributes", @aligned row); this library instead checks every
// argument on the host, returns an error code without launching anything, and sends
// shapes that are not whole tiles to the masked kernels.  The tuner follows "gemm, f32",
// section "Tuning" (two stages, finalists timed over rounds under the same clocks) and the
// lab's stopwatches (settle the clock before timing; shuffle the order every round).
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <functional>
#include <map>
#include <mutex>
#include <numeric>
#include <random>
#include <sstream>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/phx.h"
#include "internal.h"

namespace {

using phx::F16Config;
using phx::SgemmConfig;

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int64_t kMaxElems = int64_t(1) << 62;

int log_level() {
    static const int level = [] {
        const char* v = std::getenv("PHX_LOG");
        return v ? std::atoi(v) : 0;
    }();
    return level;
}

// ---------------------------------------------------------------------------------------
// Per-device state: SM count, the status word, and the workspace pool.
// ---------------------------------------------------------------------------------------
struct DevState {
    bool ready = false;
    phx_status init_status = PHX_OK;
    int sm_count = 0;
    unsigned int* status = nullptr;  // device word written by kernels
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
std::map<int, DevState> g_dev;

phx_status device_state(DevState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DevState& d = g_dev[dev];
    if (!d.ready) {
        d.ready = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            d.init_status = PHX_ERR_ARCH;
        } else if (major != 10 || minor != 3) {
            d.init_status = PHX_ERR_ARCH;  // the kernels are built for sm_103a only
        } else if (cudaMalloc(&d.status, 256) != cudaSuccess ||
                   cudaMemset(d.status, 0, 256) != cudaSuccess) {
            cudaGetLastError();
            d.init_status = PHX_ERR_NOMEM;
        } else {
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof props);
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
                cudaGetLastError();
                d.init_status = PHX_ERR_NOMEM;
            } else {
                uint64_t keep = UINT64_MAX;  // keep freed workspace for reuse
                cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
            }
        }
    }
    *out = &d;
    return d.init_status;
}

// The tuning cache's name for the current device: its name with spaces as underscores, a
// colon and its SM count ("NVIDIA_GB300:152"); "none" without a usable device.  A tuned
// configuration is only ever applied on a device with the tag it was tuned on.
std::string device_tag() {
    static std::mutex mu;
    static std::map<int, std::string> tags;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return "none";
    }
    std::lock_guard<std::mutex> lock(mu);
    auto it = tags.find(dev);
    if (it != tags.end()) return it->second;
    cudaDeviceProp prop;
    std::string tag = "none";
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
        tag = prop.name;
        for (char& c : tag)
            if (c == ' ' || c == '\t') c = '_';
        tag += ":" + std::to_string(prop.multiProcessorCount);
    } else {
        cudaGetLastError();
    }
    tags[dev] = tag;
    return tag;
}

// The current SM clock of a device in MHz, read through NVML (query calls only; nothing is
// set), or -1 when NVML is not available.  Used to record the clock beside every timing of
// the tuner's second stage.
struct NvmlApi {
    bool ok = false;
    int (*get_handle_by_pci)(const char*, void**) = nullptr;
    int (*get_clock)(void*, int, unsigned int*) = nullptr;
};

const NvmlApi& nvml() {
    static NvmlApi api;
    static std::once_flag once;
    std::call_once(once, [] {
        void* h = dlopen("libnvidia-ml.so.1", RTLD_NOW | RTLD_LOCAL);
        if (h == nullptr) return;
        auto init = reinterpret_cast<int (*)()>(dlsym(h, "nvmlInit_v2"));
        api.get_handle_by_pci = reinterpret_cast<int (*)(const char*, void**)>(
            dlsym(h, "nvmlDeviceGetHandleByPciBusId_v2"));
        api.get_clock = reinterpret_cast<int (*)(void*, int, unsigned int*)>(dlsym(h, "nvmlDeviceGetClockInfo"));
        api.ok = init != nullptr && api.get_handle_by_pci != nullptr && api.get_clock != nullptr && init() == 0;
    });
    return api;
}

double sm_clock_mhz(int dev) {
    const NvmlApi& api = nvml();
    if (!api.ok) return -1.0;
    char bus[64];
    if (cudaDeviceGetPCIBusId(bus, sizeof bus, dev) != cudaSuccess) {
        cudaGetLastError();
        return -1.0;
    }
    void* handle = nullptr;
    unsigned int mhz = 0;
    constexpr int kNvmlClockSm = 1;  // nvmlClockType_t: graphics 0, SM 1, memory 2
    if (api.get_handle_by_pci(bus, &handle) != 0 || api.get_clock(handle, kNvmlClockSm, &mhz) != 0) return -1.0;
    return static_cast<double>(mhz);
}

// ---------------------------------------------------------------------------------------
// Argument checks
// ---------------------------------------------------------------------------------------
bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    if (abytes <= 0 || bbytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

phx_status validate_sizes(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return PHX_ERR_INVALID;
    if (M * K >= kMaxElems || K * N >= kMaxElems || M * N >= kMaxElems) return PHX_ERR_INVALID;
    return PHX_OK;
}

// Sizes, null and alignment checks and the C overlap rule for operands of `ab` bytes per
// element (A, B) and `cb` bytes per element (C); pointers must be aligned to their element.
phx_status validate_elems(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                          int64_t ab, int64_t cb) {
    if (validate_sizes(M, N, K) != PHX_OK) return PHX_ERR_INVALID;
    if (M == 0 || N == 0) return PHX_OK;
    auto misaligned = [](const void* p, int64_t bytes) {
        return (reinterpret_cast<uintptr_t>(p) & static_cast<uintptr_t>(bytes - 1)) != 0;
    };
    if (C == nullptr || misaligned(C, cb)) return PHX_ERR_INVALID;
    if (K > 0) {
        if (A == nullptr || B == nullptr || misaligned(A, ab) || misaligned(B, ab)) return PHX_ERR_INVALID;
        if (overlaps(A, M * K * ab, C, M * N * cb) || overlaps(B, K * N * ab, C, M * N * cb))
            return PHX_ERR_INVALID;
    }
    return PHX_OK;
}

phx_status validate(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C) {
    return validate_elems(M, N, K, A, B, C, 4, 4);
}

// ---------------------------------------------------------------------------------------
// Configurations: names, parsing, pins, the tuning cache, defaults
// ---------------------------------------------------------------------------------------
// Configurations of a variant: its compiled GEMM tiles, then "SKINNY", the kernel for few
// rows of A (gemm_skinny.cu), which takes any M as blocks of 16 rows.
int tile_configs(int variant) {
    if (variant == PHX_VARIANT_SGEMM) return phx::sgemm_num_configs();
    if (variant == PHX_VARIANT_F16TC) return phx::f16tc_num_configs();
    return -1;
}

int num_configs(int variant) {
    const int n = tile_configs(variant);
    return n < 0 ? -1 : n + 1;
}

int skinny_index(int variant) { return tile_configs(variant); }

// Largest M for which the skinny kernel is the default: measured crossovers at K = N = 4096
// on GB300 (f32: skinny 55 us against 94 us for the tiles at M = 48, 78 against 70 at M = 64;
// f16: 27 against 31 us at M = 16, 47 against 33 at M = 32, where the tensor cores win).
int64_t skinny_default_max_m(int variant) { return variant == PHX_VARIANT_SGEMM ? 48 : 16; }

// Few columns against many rows, A stored M x K: the skinny kernels run the transposed
// product, C^T = op(B)^T @ A^T, a few-row product that streams A (each row of A one
// contiguous row of the operand the kernel streams) and writes C^T transposed, which is C.
int64_t skinny_columns_max_n(int variant) { return variant == PHX_VARIANT_SGEMM ? 16 : 8; }
bool skinny_by_columns(int variant, int trans_a, int64_t M, int64_t N) {
    return !trans_a && M >= 1024 && N < M && N <= skinny_columns_max_n(variant);
}

std::string config_name(int variant, int i) {
    char buf[128];
    if (i == skinny_index(variant)) return "SKINNY";
    if (variant == PHX_VARIANT_SGEMM) {
        const SgemmConfig& c = phx::sgemm_config(i);
        std::snprintf(buf, sizeof buf, "TILE_M=%d TILE_N=%d TILE_K=%d STAGES=%d FMA2=%d", c.tile_m,
                      c.tile_n, c.tile_k, c.stages, c.fma2);
    } else {
        const F16Config& c = phx::f16tc_config(i);
        // a 256-row tile is a 2-SM pair; a 128-row tile one CTA; CONVERT_A=1 / CONVERT_B=1 the
        // kernel that rounds A / B itself
        std::snprintf(buf, sizeof buf, "TILE_M=%d TILE_N=%d TILE_K=%d STAGES=%d%s%s", c.tile_m, c.tile_n,
                      c.tile_k, c.stages, c.convert_a ? " CONVERT_A=1" : "", c.convert_b ? " CONVERT_B=1" : "");
    }
    return buf;
}

// Parse "KEY=value KEY=value ..." and return the first compiled config that matches every
// given key (TILE_M, TILE_N, TILE_K required; STAGES optional; FMA2 for the f32 variant and
// CONVERT_A, CONVERT_B for the f16 one optional, default 0), or -1.
int parse_config(int variant, const char* spec) {
    if (spec == nullptr || num_configs(variant) < 0) return -1;
    std::map<std::string, int> kv;
    std::istringstream in(spec);
    std::string tok;
    {
        std::istringstream words(spec);
        std::string w, extra;
        if (words >> w && w == "SKINNY") return (words >> extra) ? -1 : skinny_index(variant);
    }
    while (in >> tok) {
        const size_t eq = tok.find('=');
        if (eq == std::string::npos || eq == 0 || eq + 1 >= tok.size()) return -1;
        const std::string key = tok.substr(0, eq);
        const std::string val = tok.substr(eq + 1);
        char* end = nullptr;
        const long v = std::strtol(val.c_str(), &end, 10);
        if (end == nullptr || *end != '\0') return -1;
        if (key != "TILE_M" && key != "TILE_N" && key != "TILE_K" && key != "STAGES" && key != "FMA2" &&
            key != "CONVERT_A" && key != "CONVERT_B")
            return -1;
        if (variant == PHX_VARIANT_F16TC && key == "FMA2") return -1;
        if (variant == PHX_VARIANT_SGEMM && (key == "CONVERT_A" || key == "CONVERT_B")) return -1;
        kv[key] = static_cast<int>(v);
    }
    if (!kv.count("TILE_M") || !kv.count("TILE_N") || !kv.count("TILE_K")) return -1;
    const int n = tile_configs(variant);
    for (int i = 0; i < n; ++i) {
        int tm, tn, tk, st, f2 = 0, cv = 0, cvb = 0;
        if (variant == PHX_VARIANT_SGEMM) {
            const SgemmConfig& c = phx::sgemm_config(i);
            tm = c.tile_m; tn = c.tile_n; tk = c.tile_k; st = c.stages; f2 = c.fma2;
        } else {
            const F16Config& c = phx::f16tc_config(i);
            tm = c.tile_m; tn = c.tile_n; tk = c.tile_k; st = c.stages; cv = c.convert_a; cvb = c.convert_b;
        }
        if (kv["TILE_M"] != tm || kv["TILE_N"] != tn || kv["TILE_K"] != tk) continue;
        if (kv.count("STAGES") && kv["STAGES"] != st) continue;
        if (kv.count("FMA2") && kv["FMA2"] != f2) continue;
        if (!kv.count("FMA2") && variant == PHX_VARIANT_SGEMM && f2 != 0) continue;
        if ((kv.count("CONVERT_A") ? kv["CONVERT_A"] : 0) != cv) continue;
        if ((kv.count("CONVERT_B") ? kv["CONVERT_B"] : 0) != cvb) continue;
        return i;
    }
    return -1;
}

// Tuned configurations by (device tag, variant, M, N, K).
using ShapeKey = std::tuple<std::string, int, int64_t, int64_t, int64_t>;
std::map<ShapeKey, int> g_tuned;  // guarded by g_mu
// Pinned configuration per variant: -1 none, kBadPin for an unparsable PHX_CONFIG_* (every
// call of that variant then returns PHX_ERR_CONFIG until phx_set_config replaces the pin).
constexpr int kBadPin = phx::kBadConfigPin;
int g_pin[2] = {-1, -1};          // guarded by g_mu
bool g_env_done = false;

phx_status tune_cache_read(const char* path, std::map<ShapeKey, int>* out);

void load_env_once_locked() {
    if (g_env_done) return;
    g_env_done = true;
    const char* names[2] = {"PHX_CONFIG_SGEMM", "PHX_CONFIG_F16TC"};
    for (int v = 0; v < 2; ++v) {
        const char* s = std::getenv(names[v]);
        if (s == nullptr) continue;
        g_pin[v] = parse_config(v, s);
        if (g_pin[v] < 0) {
            g_pin[v] = kBadPin;
            std::fprintf(stderr, "[phx] %s=\"%s\" names no compiled configuration; calls of this variant "
                                 "return PHX_ERR_CONFIG until phx_set_config replaces the pin\n", names[v], s);
        }
    }
    // PHX_TUNE_CACHE: a tuning cache file read at the first call (and written by phx_autotune)
    if (const char* path = std::getenv("PHX_TUNE_CACHE")) {
        std::map<ShapeKey, int> loaded;
        std::ifstream probe(path);
        if (probe) {
            probe.close();
            if (tune_cache_read(path, &loaded) == PHX_OK)
                for (const auto& kv : loaded) g_tuned[kv.first] = kv.second;
            else
                std::fprintf(stderr, "[phx] PHX_TUNE_CACHE=%s does not parse; it is ignored\n", path);
        }
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Defaults when nothing is pinned or tuned: the largest tile that still gives every SM
// work (the trade-off "gemm, f32" section "Tuning" describes: larger tiles reuse more,
// but leave fewer CTAs to spread over the card).
int default_tile_config(int variant, int64_t M, int64_t N, int64_t K, int sms, bool convert = true);
int default_config(int variant, int64_t M, int64_t N, int64_t K, int sms, bool convert = true, bool a_rows = true);

// The kernel that rounds B itself is the f16 default for few rows and a large B (see
// default_tile_config); it beats the skinny kernel from about 12 rows (measured on GB300,
// queued calls, K = N = 4096: 20.9 us against 27.0 at M = 12, 16.7 against 20.9 at M = 8).
bool f16_convert_b_fits(int64_t M, int64_t N, int64_t K) {
    return M <= 256 && N >= 1024 && static_cast<double>(K) * static_cast<double>(N) >= 8388608.0;
}

// f32 problems the skinny kernel also takes, beyond few rows: small ones, where its one
// launch and its K slices beat the tiles' grid, and 64 rows against a B that L2 holds while
// the four 16-row chunks read it (measured on GB300, queued calls: 256^3 8.3 us against 14.5
// with 64 x 64 tiles, 384^3 10.4 against 14.5, (128, 1024, 1024) 16.5 against 18.7,
// (64, 2048, 2048) 24.7 against 39.2; 512^3 16.5 against 16.6; 768^3 37.0 against 31.4).
bool sgemm_skinny_fits(int64_t M, int64_t N, int64_t K) {
    const double mnk = static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
    const double kn = static_cast<double>(K) * static_cast<double>(N);
    return (M <= 512 && mnk <= 134217728.0) || (M <= 64 && kn <= 4194304.0);
}

// a_rows: A is stored M x K (the skinny kernels' few-columns form needs that).
int default_config(int variant, int64_t M, int64_t N, int64_t K, int sms, bool convert, bool a_rows) {
    const bool skip_skinny = variant == PHX_VARIANT_F16TC && convert && M > 8 && f16_convert_b_fits(M, N, K);
    if (M <= skinny_default_max_m(variant) && !skip_skinny) return skinny_index(variant);
    // Few columns, an A of 2^22 elements or more: one pass over A.  For f16, where the kernel
    // that rounds A inside the GEMM takes over (A of 2^23 elements or more), only up to 4
    // columns and 4096 rows.  Measured on GB300, queued calls, K = 4096: f32 N = 1 12.4 us
    // against 88.2 with tiles, N = 8 26.8 against 78.1, N = 16 45.2 against 78.1, (16384, 8,
    // 4096) 90 against 230; f16 (4096, 1, 4096) 14.5 against 22.7 for the kernel that rounds A,
    // N = 4 20.6 against 22.6, but N = 8 28.8 against 22.7 and (16384, 8, 4096) 100.7 against
    // 57.0; (1024, 4, 4096) 10.4 against 18.3 for the kernel that rounds both.
    const double mk = static_cast<double>(M) * static_cast<double>(K);
    if (a_rows && skinny_by_columns(variant, 0, M, N) && mk >= 4194304.0 &&
        (variant == PHX_VARIANT_SGEMM || mk < 8388608.0 || (N <= 4 && M <= 4096)))
        return skinny_index(variant);
    if (variant == PHX_VARIANT_SGEMM && sgemm_skinny_fits(M, N, K)) return skinny_index(variant);
    return default_tile_config(variant, M, N, K, sms, convert);
}

// The compiled configurations the defaults name, resolved once (parsing a name per call
// would cost a microsecond of host time).
struct DefaultConfigs {
    int s128x128 = -1, s128x64 = -1, s64x64 = -1, s64x128 = -1, s128x64f2 = -1;  // f32
    int t256x256 = -1, t128x256 = -1, t128x128 = -1, t128x64 = -1;  // f16 tensor cores
    int c64 = -1, c128 = -1, c256 = -1;  // f16, A rounded in the kernel, TILE_N = 64, 128, 256
    int cb64 = -1, cb128 = -1;           // f16, B rounded in the kernel, TILE_N = 64, 128
    int cab64 = -1;                      // f16, both rounded in the kernel, TILE_N = 64
};

const DefaultConfigs& default_configs() {
    static const DefaultConfigs d = [] {
        DefaultConfigs c;
        c.s128x128 = parse_config(PHX_VARIANT_SGEMM, "TILE_M=128 TILE_N=128 TILE_K=16 STAGES=4 FMA2=1");
        c.s128x64 = parse_config(PHX_VARIANT_SGEMM, "TILE_M=128 TILE_N=64 TILE_K=8 STAGES=4");
        c.s64x64 = parse_config(PHX_VARIANT_SGEMM, "TILE_M=64 TILE_N=64 TILE_K=8 STAGES=4");
        c.s64x128 = parse_config(PHX_VARIANT_SGEMM, "TILE_M=64 TILE_N=128 TILE_K=16 STAGES=4 FMA2=1");
        c.s128x64f2 = parse_config(PHX_VARIANT_SGEMM, "TILE_M=128 TILE_N=64 TILE_K=16 STAGES=4 FMA2=1");
        c.t256x256 = parse_config(PHX_VARIANT_F16TC, "TILE_M=256 TILE_N=256 TILE_K=64 STAGES=6");
        c.t128x256 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=256 TILE_K=64 STAGES=4");
        c.t128x128 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=128 TILE_K=64 STAGES=6");
        c.t128x64 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=64 TILE_K=64 STAGES=8");
        c.c64 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=64 TILE_K=64 STAGES=4 CONVERT_A=1");
        c.c128 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=128 TILE_K=64 STAGES=3 CONVERT_A=1");
        c.c256 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=256 TILE_K=64 STAGES=2 CONVERT_A=1");
        c.cb64 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=64 TILE_K=64 STAGES=4 CONVERT_B=1");
        c.cb128 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=128 TILE_K=64 STAGES=3 CONVERT_B=1");
        c.cab64 = parse_config(PHX_VARIANT_F16TC, "TILE_M=128 TILE_N=64 TILE_K=64 STAGES=3 CONVERT_A=1 CONVERT_B=1");
        return c;
    }();
    return d;
}

// Problems of at most this many multiply-adds (2^28: 512 x 512 x 1024) take the small f32
// tiles: their time is the latency of a few k steps, and more, smaller CTAs spread it over
// more SMs (measured on GB300, queued calls: 512^3 16.5 us with 128 x 64 tiles against 22.8
// with 128 x 128; 256^3 14.4 us with 64 x 64 against 22.7).
constexpr int64_t kSmallSgemmWork = int64_t(1) << 28;

// With `convert`, the f16 default may be the kernel that rounds A or B itself; callers whose
// operands are not row-major f32 matrices pass false.
int default_tile_config(int variant, int64_t M, int64_t N, int64_t K, int sms, bool convert) {
    const DefaultConfigs& dc = default_configs();
    if (variant == PHX_VARIANT_SGEMM) {
        const int64_t slots = 2 * static_cast<int64_t>(sms);  // two CTAs per SM
        if (static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) <=
            static_cast<double>(kSmallSgemmWork))
            return ceil_div(M, 128) * ceil_div(N, 64) >= 32 ? dc.s128x64 : dc.s64x64;
        // 128 x 128 tiles whenever they exist: a grid too small for the GPU is then spread as
        // stream-K blocks or split along K, which keeps the larger, more efficient tile
        if (M >= 128 && N >= 128) return dc.s128x128;
        // fewer than 128 rows against 128 columns or more: 128-row tiles from 65 rows on, 64 x 128
        // tiles below (measured on GB300, queued calls, K = N = 4096: M = 96 98.9 us against
        // 134.5 with 64 x 64 tiles; M = 64 62.4 against 74.5; (64, 8192, 4096) 104 against 141)
        if (N >= 128) return M > 64 ? dc.s128x128 : dc.s64x128;
        // ... and the same across: 128 rows or more against fewer than 128 columns ((4096, 64,
        // 4096) 64.0 us against 74.5; (4096, 96, 4096) 99.0 against 137.9; (8192, 32, 4096)
        // 108.3 against 138.3)
        if (M >= 128) return N > 64 ? dc.s128x128 : dc.s128x64f2;
        if (ceil_div(M, 128) * ceil_div(N, 128) >= slots) return dc.s128x128;
        if (ceil_div(M, 128) * ceil_div(N, 64) >= slots) return dc.s128x64;
        return dc.s64x64;
    }
    // Few columns, many rows: A is most of the bytes, and rounding it inside the GEMM saves
    // writing and reading back its f16 copy.  One tile of N, and 128-row tiles for at least
    // half the SMs; or fewer row tiles, with K split to give every SM work, where the copy
    // saved outweighs the split's extra launch and planes: A of 2^23 elements or more, and
    // K >= 2048.  Measured on GB300, queued calls: (4096, 128, 4096) 25.1 us against 33.1 for
    // the other kernel, (8192, 128, 4096) 42.2 against 53.7, (2048, 128, 4096) 19.0 against
    // 20.9, (8192, 64, 2048) 22.9 against 27.9; but (4096, 128, 1024) 18.7 against about 13.
    if (convert && N <= 256 &&
        (ceil_div(M, 128) >= sms / 2 || (M >= 1024 && K >= 2048 && M * K >= (int64_t(1) << 23))))
        return N <= 64 ? dc.c64 : N <= 128 ? dc.c128 : dc.c256;
    // Few rows, a large B (2^23 elements or more): B is most of the bytes; the kernel rounds
    // B itself, and splits K to give every SM work.  (Few enough rows take the skinny kernel
    // before this.)  Measured on GB300, queued calls: (64, 4096, 4096) 21.1 us against 32.9
    // for the best tile of the other kernel, (64, 8192, 8192) 55 against 105; with a small B,
    // (64, 1024, 1024), 16.6 against 12.7.
    if (convert && f16_convert_b_fits(M, N, K)) return dc.cb128;
    // Tiny problems (2^25 multiply-adds or fewer): both operands rounded in the kernel, one
    // launch and no scratch (measured on GB300, synced calls: 256^3 15.5 us against 17.3 for
    // the rounding pass and the 128 x 128 tile; even at 512^3, slower from 768^3 on, where
    // every tile rounding its own A and B boxes costs more than one pass).
    if (convert && static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) <= 33554432.0)
        return dc.cab64;
    if (M >= 256 && N >= 256) {
        // the 2-SM 256 x 256 tile when it fills the CTA pairs, or when a grid too small for
        // the GPU is split along K (32 or more k blocks of 64); else the one-CTA tile that gives more
        // SMs work (measured on GB300, queued calls: 2048^3 24.8 us with 128 x 256 against
        // 26.3 with 2-SM 256 x 256 on 128 SMs; 1024^3 14.4 against 16.5; 512^3 10.4 against
        // 12.5)
        const int64_t pairs = ceil_div(M, 256) * ceil_div(N, 256);
        const int64_t workers = sms / 2;
        const bool k_split = 2 * pairs <= workers && ceil_div(K, 64) >= 32;
        if (pairs >= workers || k_split) return dc.t256x256;
        if (ceil_div(M, 128) * ceil_div(N, 256) >= 3 * static_cast<int64_t>(sms) / 4) return dc.t128x256;
        return dc.t128x128;
    }
    if (ceil_div(M, 128) * ceil_div(N, 256) >= sms) return dc.t128x256;
    if (ceil_div(M, 128) * ceil_div(N, 128) >= sms) return dc.t128x128;
    return dc.t128x64;
}

// The configuration for a call: the pin, else the tuned one for this device and shape, else
// the default; kBadPin when the variant's PHX_CONFIG_* pin does not parse.
int choose_config(int variant, int64_t M, int64_t N, int64_t K, int sms, int trans_a = 0) {
    const std::string tag = device_tag();
    std::lock_guard<std::mutex> lock(g_mu);
    load_env_once_locked();
    if (g_pin[variant] >= 0 || g_pin[variant] == kBadPin) return g_pin[variant];
    auto it = g_tuned.find(ShapeKey(tag, variant, M, N, K));
    if (it != g_tuned.end()) return it->second;
    return default_config(variant, M, N, K, sms, true, !trans_a);
}

phx_status config_error(int cfg) { return cfg == kBadPin ? PHX_ERR_CONFIG : PHX_ERR_INTERNAL; }

// The last tuning run's report per variant (phx_autotune_report); guarded by g_mu.
std::string g_tune_report[2];

// Tuning cache file: "# ..." comments, then one line per entry:
//   <device tag> <variant> <M> <N> <K> <configuration name>
// Entries of every device are kept; a call only uses those of its own device's tag.
phx_status tune_cache_write_locked(const char* path) {
    std::ofstream f(path);
    if (!f) return PHX_ERR_INVALID;
    f << "# phx tuning cache: device variant M N K config\n";
    for (const auto& kv : g_tuned) {
        f << std::get<0>(kv.first) << ' ' << std::get<1>(kv.first) << ' ' << std::get<2>(kv.first) << ' '
          << std::get<3>(kv.first) << ' ' << std::get<4>(kv.first) << ' '
          << config_name(std::get<1>(kv.first), kv.second) << '\n';
    }
    return f ? PHX_OK : PHX_ERR_INVALID;
}

phx_status tune_cache_read(const char* path, std::map<ShapeKey, int>* out) {
    std::ifstream f(path);
    if (!f) return PHX_ERR_INVALID;
    std::string line;
    while (std::getline(f, line)) {
        if (line.empty() || line[0] == '#') continue;
        std::istringstream in(line);
        std::string tag;
        int variant;
        long long M, N, K;
        if (!(in >> tag >> variant >> M >> N >> K)) return PHX_ERR_CONFIG;
        if (tag.find(':') == std::string::npos && tag != "none") return PHX_ERR_CONFIG;
        std::string rest;
        std::getline(in, rest);
        if (num_configs(variant) < 0) return PHX_ERR_CONFIG;
        const int idx = parse_config(variant, rest.c_str());
        if (idx < 0) return PHX_ERR_CONFIG;
        (*out)[ShapeKey(tag, variant, M, N, K)] = idx;
    }
    return PHX_OK;
}

// The configuration the last GEMM call of each variant launched (-1: none yet), for reports.
std::atomic<int> g_last_cfg[2] = {{-1}, {-1}};

// ---------------------------------------------------------------------------------------
// The tuner's selection logic, shared by phx_autotune and phx_selftest_tuner.
// measure(i) returns the seconds one launch of candidate i took, or a negative value if
// the candidate failed (it is then dropped); elapsed() is the clock the settle phase uses.
// ---------------------------------------------------------------------------------------
struct TuneOutcome {
    int picked = -1;
    int64_t launches = 0;
};

double median(std::vector<double> v) {
    std::sort(v.begin(), v.end());
    const size_t n = v.size();
    return n == 0 ? 0.0 : (n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]));
}

TuneOutcome tune_select(int n, const std::function<double(int)>& measure,
                        const std::function<double()>& elapsed, int finalists, int rounds,
                        double settle_s, uint64_t seed,
                        const std::function<void(int, double)>& stage2_timed = nullptr) {
    TuneOutcome out;
    auto run = [&](int i) {
        ++out.launches;
        return measure(i);
    };
    // Stage 1: every candidate, one warm-up launch and three timed ones; failures dropped.
    std::vector<std::pair<double, int>> scored;
    for (int i = 0; i < n; ++i) {
        if (run(i) < 0) continue;
        std::vector<double> t;
        bool failed = false;
        for (int r = 0; r < 3 && !failed; ++r) {
            const double s = run(i);
            if (s < 0) failed = true;
            t.push_back(s);
        }
        if (!failed) scored.emplace_back(median(t), i);
    }
    if (scored.empty()) return out;
    std::sort(scored.begin(), scored.end());
    const int k = std::max(1, std::min<int>(finalists, static_cast<int>(scored.size())));
    std::vector<int> fin;
    for (int j = 0; j < k; ++j) fin.push_back(scored[j].second);
    // Stage 2a: settle the clocks on the finalists' own work.
    const double t0 = elapsed();
    while (elapsed() - t0 < settle_s)
        for (int i : fin) run(i);
    // Stage 2b: `rounds` rounds, one launch of each finalist per round, shuffled each round.
    std::mt19937_64 rng(seed);
    std::map<int, std::vector<double>> times;
    std::map<int, bool> dropped;
    for (int r = 0; r < std::max(1, rounds); ++r) {
        std::vector<int> order = fin;
        std::shuffle(order.begin(), order.end(), rng);
        for (int i : order) {
            if (dropped[i]) continue;
            const double s = run(i);
            if (s < 0) {
                dropped[i] = true;
            } else {
                times[i].push_back(s);
                if (stage2_timed) stage2_timed(i, s);
            }
        }
    }
    double best = 0.0;
    for (int i : fin) {
        if (dropped[i] || times[i].empty()) continue;
        const double m = median(times[i]);
        if (out.picked < 0 || m < best) {
            best = m;
            out.picked = i;
        }
    }
    return out;
}

// Fill n floats with small values (uniform-ish in [-1, 1)) for the tuner's scratch inputs.
__global__ void tune_fill_kernel(float* p, int64_t n, uint32_t salt) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        uint32_t h = static_cast<uint32_t>(i) * 2654435761u ^ salt;
        h ^= h >> 15;
        h *= 2246822519u;
        h ^= h >> 13;
        p[i] = static_cast<float>(h >> 8) * (1.0f / 8388608.0f) - 1.0f;
    }
}

// ---------------------------------------------------------------------------------------
// Per-kernel timing (phx_profile_start / phx_profile_stop): events recorded on the call's
// stream around every kernel the library launches, summed per kernel kind at stop.
// ---------------------------------------------------------------------------------------
enum KernelKind { kKindSgemm = 0, kKindCast = 1, kKindTcGemm = 2, kKindScale = 3, kKindTranspose = 4,
                  kKindSkinny = 5, kNumKinds = 6 };

thread_local int64_t t_launches = 0;

struct Profile {
    bool on = false;
    std::vector<std::tuple<int, cudaEvent_t, cudaEvent_t, int64_t>> marks;  // kind, begin, end, kernels
    std::vector<cudaEvent_t> spare;
};
std::mutex g_prof_mu;
Profile g_prof;

cudaEvent_t prof_event() {
    if (!g_prof.spare.empty()) {
        cudaEvent_t e = g_prof.spare.back();
        g_prof.spare.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Runs `launch` on `stream`, bracketed by events when profiling is on.
template <class F>
cudaError_t timed(int kind, cudaStream_t stream, F&& launch) {
    std::unique_lock<std::mutex> lock(g_prof_mu);
    if (!g_prof.on) {
        lock.unlock();
        return launch();
    }
    cudaEvent_t b = prof_event(), e = prof_event();
    cudaEventRecord(b, stream);
    const int64_t n0 = t_launches;
    const cudaError_t err = launch();
    cudaEventRecord(e, stream);
    g_prof.marks.emplace_back(kind, b, e, t_launches - n0);
    return err;
}

// An f32 operand given transposed is copied into its plain layout first (pooled scratch);
// the copies start on 256-byte boundaries so that the aligned kernels apply whenever the
// shape allows.
phx_status launch_sgemm_transposed(int cfg, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                   float alpha, const float* A, const float* B, float beta, float* C,
                                   DevState* d, cudaStream_t stream);

phx_status launch_skinny(int variant, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                         float alpha, const float* A, const float* B, float beta, float* C,
                         DevState* d, cudaStream_t stream) {
    const size_t bytes = phx::skinny_run_bytes(variant, trans_a, trans_b, M, N, K, A, B, d->sm_count);
    void* ws = nullptr;
    if (bytes > 0 && cudaMallocFromPoolAsync(&ws, bytes, d->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_NOMEM;
    }
    const cudaError_t err = timed(kKindSkinny, stream, [&] {
        return phx::skinny_run(variant, trans_a, trans_b, M, N, K, alpha, A, B, beta, C, ws, d->sm_count, stream);
    });
    if (ws != nullptr) cudaFreeAsync(ws, stream);
    return err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

// A large f32 problem whose rows of A or B do not start on 16 bytes (K % 4 != 0, N % 4 != 0,
// or an unaligned base) would be copied 4 bytes at a time.  Instead, A (when K % 4 != 0 or A
// is unaligned) is copied into M x Kp and B into Kp x Np (Kp, Np: K, N rounded up to a
// multiple of 4), zeros in the new columns and rows, in pooled scratch; the 16-byte-copy
// kernel then runs on (M, N, Kp) with B's rows Np apart and writes C in place (4-byte stores
// when C's rows are not 16-byte aligned).  The zeros add exact zeros, so the result is the
// same (up to the sign of a zero sum), for two copies of A and B (about 2 % of a 4096-class
// GEMM).
phx_status launch_sgemm_padded(int cfg, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                               const float* B, float beta, float* C, DevState* d, cudaStream_t stream) {
    auto r256 = [](int64_t b) { return (b + 255) / 256 * 256; };
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const int64_t Kp = (K + 3) / 4 * 4, Np = (N + 3) / 4 * 4;
    const bool pad_a = K % 4 != 0 || !al16(A);
    const bool pad_b = K % 4 != 0 || N % 4 != 0 || !al16(B);
    const int64_t a_bytes = pad_a ? r256(M * Kp * 4) : 0;
    const int64_t b_bytes = pad_b ? r256(Kp * Np * 4) : 0;
    const float* Ap = A;
    const float* Bp = B;
    const int64_t ldb = pad_b ? Np : N;
    // the stream-K or split-K scratch of the padded problem follows the copies
    const size_t sk_bytes = phx::sgemm_workspace_bytes(cfg, M, N, Kp, reinterpret_cast<const float*>(256),
                                                       reinterpret_cast<const float*>(256), C, d->sm_count, ldb);
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(a_bytes + b_bytes) + sk_bytes, d->pool, stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_NOMEM;
    }
    cudaError_t err = cudaSuccess;
    if (pad_a) {
        float* Ad = static_cast<float*>(ws);
        err = timed(kKindTranspose, stream,
                    [&] { return phx::pad_copy_launch(A, M, K, K, Ad, M, Kp, d->sm_count, stream); });
        Ap = Ad;
    }
    if (err == cudaSuccess && pad_b) {
        float* Bd = reinterpret_cast<float*>(static_cast<char*>(ws) + a_bytes);
        err = timed(kKindTranspose, stream,
                    [&] { return phx::pad_copy_launch(B, K, N, N, Bd, Kp, Np, d->sm_count, stream); });
        Bp = Bd;
    }
    if (err == cudaSuccess) {
        void* sk_ws = sk_bytes > 0 ? static_cast<char*>(ws) + a_bytes + b_bytes : nullptr;
        err = timed(kKindSgemm, stream, [&] {
            return phx::sgemm_launch(cfg, M, N, Kp, alpha, Ap, Bp, beta, C, sk_ws, d->sm_count, stream, ldb);
        });
    }
    cudaFreeAsync(ws, stream);
    return err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

phx_status launch_variant(int variant, int cfg, int64_t M, int64_t N, int64_t K, float alpha,
                          const float* A, const float* B, float beta, float* C, DevState* d,
                          cudaStream_t stream, int trans_a = 0, int trans_b = 0) {
    // the kernel that rounds A (B) reads A stored M x K (B stored K x N) only: an operand
    // given transposed takes the default without that kernel (the skinny kernel included)
    if (variant == PHX_VARIANT_F16TC &&
        ((trans_a && phx::f16tc_is_convert_a(cfg)) || (trans_b && phx::f16tc_is_convert_b(cfg)))) {
        cfg = default_config(PHX_VARIANT_F16TC, M, N, K, d->sm_count, false, !trans_a);
        g_last_cfg[PHX_VARIANT_F16TC].store(cfg);
    }
    if (cfg == skinny_index(variant))
        return launch_skinny(variant, trans_a, trans_b, M, N, K, alpha, A, B, beta, C, d, stream);
    if (variant == PHX_VARIANT_SGEMM && (trans_a || trans_b))
        return launch_sgemm_transposed(cfg, trans_a, trans_b, M, N, K, alpha, A, B, beta, C, d, stream);
    if (variant == PHX_VARIANT_SGEMM && phx::sgemm_scalar_edge(cfg, M, N, K, A, B, C) && M >= 512 && N >= 512 &&
        M * N * K >= (int64_t(1) << 32))
        return launch_sgemm_padded(cfg, M, N, K, alpha, A, B, beta, C, d, stream);
    if (variant == PHX_VARIANT_SGEMM) {
        // pooled scratch only for a stream-K spread or a grid split along K
        const size_t bytes = phx::sgemm_workspace_bytes(cfg, M, N, K, A, B, C, d->sm_count);
        void* ws = nullptr;
        if (bytes > 0 && cudaMallocFromPoolAsync(&ws, bytes, d->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return PHX_ERR_NOMEM;
        }
        const cudaError_t err = timed(kKindSgemm, stream, [&] {
            return phx::sgemm_launch(cfg, M, N, K, alpha, A, B, beta, C, ws, d->sm_count, stream);
        });
        if (ws != nullptr) cudaFreeAsync(ws, stream);
        return err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
    }
    // one pooled block holds the call's scratch (phx::f16tc_run_bytes; none for the kernel
    // that rounds both operands without a split)
    const size_t bytes = phx::f16tc_run_bytes(cfg, M, N, K, d->sm_count);
    void* ws = nullptr;
    if (bytes > 0 && cudaMallocFromPoolAsync(&ws, bytes, d->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_NOMEM;
    }
    const cudaError_t err = phx::f16tc_run(cfg, trans_a, trans_b, M, N, K, alpha, A, B, beta, C, ws, d->status,
                                           d->sm_count, stream);
    if (ws != nullptr) cudaFreeAsync(ws, stream);
    return err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

phx_status launch_sgemm_transposed(int cfg, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                   float alpha, const float* A, const float* B, float beta, float* C,
                                   DevState* d, cudaStream_t stream) {
    auto r256 = [](int64_t b) { return (b + 255) / 256 * 256; };
    const int64_t a_bytes = trans_a ? r256(M * K * 4) : 0;
    const int64_t b_bytes = trans_b ? r256(K * N * 4) : 0;
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(a_bytes + b_bytes), d->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_NOMEM;
    }
    float* At = trans_a ? static_cast<float*>(ws) : nullptr;
    float* Bt = trans_b ? reinterpret_cast<float*>(static_cast<char*>(ws) + a_bytes) : nullptr;
    cudaError_t err = cudaSuccess;
    if (trans_a)  // A stored K x M
        err = timed(kKindTranspose, stream, [&] { return phx::transpose_f32_launch(A, At, K, M, stream); });
    if (err == cudaSuccess && trans_b)  // B stored N x K
        err = timed(kKindTranspose, stream, [&] { return phx::transpose_f32_launch(B, Bt, N, K, stream); });
    phx_status st = err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
    if (st == PHX_OK)
        st = launch_variant(PHX_VARIANT_SGEMM, cfg, M, N, K, alpha, trans_a ? At : A, trans_b ? Bt : B, beta,
                            C, d, stream);
    cudaFreeAsync(ws, stream);
    return st;
}

phx_status gemm_entry(int variant, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                      const float* B, float beta, float* C, cudaStream_t stream, int trans_a = 0,
                      int trans_b = 0) {
    phx_status st = validate(M, N, K, A, B, C);
    if (st != PHX_OK) return st;
    if (M == 0 || N == 0) return PHX_OK;
    DevState* d = nullptr;
    st = device_state(&d);
    if (st != PHX_OK) return st;
    if (K == 0 || alpha == 0.f) {
        if (beta == 1.f) return PHX_OK;
        return timed(kKindScale, stream, [&] { return phx::scale_c_launch(M, N, beta, C, stream); }) ==
                       cudaSuccess
                   ? PHX_OK : PHX_ERR_LAUNCH;
    }
    const int cfg = choose_config(variant, M, N, K, d->sm_count, trans_a);
    if (cfg < 0) return config_error(cfg);
    g_last_cfg[variant].store(cfg);
    if (log_level() >= 2)
        std::fprintf(stderr, "[phx] variant %d (%lld,%lld,%lld): %s\n", variant, (long long)M,
                     (long long)N, (long long)K, config_name(variant, cfg).c_str());
    return launch_variant(variant, cfg, M, N, K, alpha, A, B, beta, C, d, stream, trans_a, trans_b);
}

// Half-precision operands (phx_gemm_f16in_*): no rounding pass, only the copy into the
// K-major layout the tensor cores read, which A skips when it can be read in place (stored
// M x K with K a multiple of 8 and 16-byte aligned).  The tile configuration is the f16
// variant's; where that would be the skinny kernel, which reads f32, the default tile.
phx_status f16in_entry(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                       const void* B, float beta, float* C, __half* Ch, cudaStream_t stream) {
    phx_status st = validate_elems(M, N, K, A, B, C != nullptr ? static_cast<const void*>(C) : Ch, 2,
                                   C != nullptr ? 4 : 2);
    if (st != PHX_OK) return st;
    if (M == 0 || N == 0) return PHX_OK;
    DevState* d = nullptr;
    st = device_state(&d);
    if (st != PHX_OK) return st;
    if (K == 0 || alpha == 0.f) {
        if (beta == 1.f) return PHX_OK;
        const cudaError_t err = timed(kKindScale, stream, [&] {
            return C != nullptr ? phx::scale_c_launch(M, N, beta, C, stream) : phx::scale_c_h_launch(M, N, beta, Ch, stream);
        });
        return err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
    }
    int cfg = choose_config(PHX_VARIANT_F16TC, M, N, K, d->sm_count);
    // the skinny kernel and the kernel that rounds A read f32 operands: the default tile then
    if (cfg == skinny_index(PHX_VARIANT_F16TC) || (cfg >= 0 && phx::f16tc_is_convert(cfg)))
        cfg = default_tile_config(PHX_VARIANT_F16TC, M, N, K, d->sm_count, false);
    if (cfg < 0) return config_error(cfg);
    g_last_cfg[PHX_VARIANT_F16TC].store(cfg);
    const int64_t Kp = (K + 7) / 8 * 8;
    const bool a_direct = !trans_a && K % 8 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0;
    auto r256 = [](int64_t b) { return (b + 255) / 256 * 256; };
    const int64_t a_bytes = a_direct ? 0 : r256(M * Kp * 2);
    const int64_t b_bytes = r256(N * Kp * 2);
    const size_t split_bytes = phx::f16tc_split_bytes(cfg, M, N, K, d->sm_count);
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(a_bytes + b_bytes) + split_bytes, d->pool, stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_NOMEM;
    }
    __half* Ah = a_direct ? nullptr : static_cast<__half*>(ws);
    __half* Bt = reinterpret_cast<__half*>(static_cast<char*>(ws) + a_bytes);
    void* split_ws = split_bytes > 0 ? static_cast<char*>(ws) + a_bytes + b_bytes : nullptr;
    cudaError_t err = timed(kKindCast, stream, [&] {
        return phx::f16tc_prepare_launch(1, trans_a, trans_b, M, N, K, A, B, Ah, Bt, d->sm_count, stream);
    });
    if (err == cudaSuccess)
        err = timed(kKindTcGemm, stream, [&] {
            const __half* a_ops = a_direct ? static_cast<const __half*>(A) : Ah;
            return phx::f16tc_gemm_launch_ops(cfg, M, N, K, alpha, beta, C, Ch, a_ops, a_direct ? K : Kp, Bt, Kp,
                                              split_ws, d->status, d->sm_count, stream);
        });
    cudaFreeAsync(ws, stream);
    return err == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

bool valid_op(phx_op op) {
    const int v = static_cast<int>(op);
    return v == PHX_OP_N || v == PHX_OP_T;
}

phx_status copy_name(const std::string& s, char* buf, size_t buflen) {
    if (buf == nullptr || buflen == 0) return PHX_ERR_INVALID;
    if (s.size() + 1 > buflen) return PHX_ERR_INVALID;
    std::memcpy(buf, s.c_str(), s.size() + 1);
    return PHX_OK;
}

}  // namespace

namespace phx {
// The skinny kernels read A in either storage order; B stored transposed (N x K) has a
// kernel of its own, which streams B's rows; few columns against many rows, with A stored
// M x K, run as the transposed product on that kernel, streaming A's rows
// (skinny_by_columns).
size_t skinny_run_bytes(int variant, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, const float* A,
                        const float* B, int num_sms) {
    const int f16 = variant == PHX_VARIANT_F16TC ? 1 : 0;
    if (skinny_by_columns(variant, trans_a, M, N)) return skinny_nt_workspace_bytes(f16, N, M, K, A, num_sms);
    return trans_b ? skinny_nt_workspace_bytes(f16, M, N, K, B, num_sms)
                   : skinny_workspace_bytes(f16, M, N, K, B, num_sms);
}

cudaError_t skinny_run(int variant, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, float alpha,
                       const float* A, const float* B, float beta, float* C, void* ws, int num_sms,
                       cudaStream_t stream) {
    const int f16 = variant == PHX_VARIANT_F16TC ? 1 : 0;
    if (skinny_by_columns(variant, trans_a, M, N))
        // C^T (N x M) = op(B)^T @ A^T: the few rows are op(B)^T, which is B stored transposed
        // (B stored K x N) or plain (B stored N x K); A (M x K) is the streamed operand; C^T
        // written transposed is C
        return skinny_nt_launch(f16, trans_b ? 0 : 1, N, M, K, alpha, B, A, beta, C, ws, num_sms, stream, 1);
    return trans_b ? skinny_nt_launch(f16, trans_a, M, N, K, alpha, A, B, beta, C, ws, num_sms, stream)
                   : skinny_launch(f16, trans_a, M, N, K, alpha, A, B, beta, C, ws, num_sms, stream);
}

size_t f16tc_run_bytes(int cfg, int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t Kp = (K + 7) / 8 * 8;
    // the kernel that rounds both itself: only the partial planes of a split along K; A (B)
    // itself: B's (A's) f16 copy, then the planes
    if (f16tc_is_convert_a(cfg) && f16tc_is_convert_b(cfg)) return f16tc_split_bytes(cfg, M, N, K, num_sms);
    if (f16tc_is_convert_a(cfg))
        return static_cast<size_t>((N * Kp * 2 + 255) / 256 * 256) + f16tc_split_bytes(cfg, M, N, K, num_sms);
    if (f16tc_is_convert_b(cfg))
        return static_cast<size_t>((M * Kp * 2 + 255) / 256 * 256) + f16tc_split_bytes(cfg, M, N, K, num_sms);
    // the f16 operand copies, then (for a grid split along K) the partial products of the
    // slices
    return f16tc_workspace_bytes(M, N, K) + f16tc_split_bytes(cfg, M, N, K, num_sms);
}

cudaError_t f16tc_run(int cfg, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, float alpha,
                      const float* A, const float* B, float beta, float* C, void* ws, unsigned int* status,
                      int num_sms, cudaStream_t stream) {
    if (f16tc_is_convert(cfg)) {
        // The other operand's f16 copy at the start of ws (B as N x Kp, or A as M x Kp), the
        // partial planes of a split after it, then the GEMM that rounds its operand as it
        // reads it (stored M x K for A, K x N for B: not transposed)
        const bool ca = f16tc_is_convert_a(cfg), cb = f16tc_is_convert_b(cfg);
        if ((ca && trans_a) || (cb && trans_b)) return cudaErrorInvalidValue;
        const int64_t Kp = (K + 7) / 8 * 8;
        const int ci = cfg - (f16tc_num_configs() - f16cvt_num_configs());
        if (ca && cb) {
            // both rounded in the kernel: one launch, scratch only for a split's planes
            void* split = f16tc_split_bytes(cfg, M, N, K, num_sms) > 0 ? ws : nullptr;
            return timed(kKindTcGemm, stream, [&] {
                return f16cvt_gemm_launch(ci, M, N, K, alpha, beta, C, A, B, nullptr, 0, split, status, num_sms,
                                          stream);
            });
        }
        __half* other = static_cast<__half*>(ws);
        // the partial planes of a split follow the other operand's copy (A's, or B's)
        void* split = f16tc_split_bytes(cfg, M, N, K, num_sms) > 0
                          ? static_cast<char*>(ws) + ((cb ? M : N) * Kp * 2 + 255) / 256 * 256
                          : nullptr;
        cudaError_t err = timed(kKindCast, stream, [&] {
            return cb ? f16tc_prepare_launch(0, trans_a, 0, M, N, K, A, B, other, nullptr, num_sms, stream)
                      : f16tc_prepare_launch(0, 0, trans_b, M, N, K, A, B, nullptr, other, num_sms, stream);
        });
        if (err == cudaSuccess)
            err = timed(kKindTcGemm, stream, [&] {
                return f16cvt_gemm_launch(ci, M, N, K, alpha, beta, C, A, B, other, Kp, split, status, num_sms,
                                          stream);
            });
        return err;
    }
    const size_t cast_bytes = f16tc_workspace_bytes(M, N, K);
    const size_t split_bytes = f16tc_split_bytes(cfg, M, N, K, num_sms);
    void* split_ws = split_bytes > 0 ? static_cast<char*>(ws) + cast_bytes : nullptr;
    cudaError_t err = timed(kKindCast, stream, [&] {
        return f16tc_cast_launch_ex(trans_a, trans_b, M, N, K, A, B, ws, num_sms, stream);
    });
    if (err == cudaSuccess)
        err = timed(kKindTcGemm, stream, [&] {
            return f16tc_gemm_launch(cfg, M, N, K, alpha, beta, C, ws, split_ws, status, num_sms, stream);
        });
    return err;
}

// The configuration a call of `variant` with this shape would use (pin, tuned, default),
// for entry points outside this file.
int choose_config_for(int variant, int64_t M, int64_t N, int64_t K, int sms) {
    return choose_config(variant, M, N, K, sms);
}

bool is_skinny_config(int variant, int cfg) { return cfg == skinny_index(variant); }
}  // namespace phx

extern "C" {

const char* phx_version(void) { return "phx 0.1 (sm_103a)"; }

const char* phx_status_string(phx_status s) {
    switch (s) {
        case PHX_OK: return "PHX_OK";
        case PHX_ERR_INVALID: return "PHX_ERR_INVALID: invalid argument";
        case PHX_ERR_ARCH: return "PHX_ERR_ARCH: no sm_103 device";
        case PHX_ERR_LAUNCH: return "PHX_ERR_LAUNCH: CUDA call or kernel launch failed";
        case PHX_ERR_TIMEOUT: return "PHX_ERR_TIMEOUT: a device-side wait gave up";
        case PHX_ERR_NOMEM: return "PHX_ERR_NOMEM: workspace allocation failed";
        case PHX_ERR_INTERNAL: return "PHX_ERR_INTERNAL: library invariant failed";
        case PHX_ERR_CONFIG: return "PHX_ERR_CONFIG: unknown or unparsable configuration";
    }
    return "unknown phx_status";
}

phx_status phx_validate_args(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                             const void* C) {
    return validate(M, N, K, A, B, C);
}

phx_status phx_sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float* A, const float* B,
                     float beta, float* C, phx_stream_t stream) {
    return gemm_entry(PHX_VARIANT_SGEMM, M, N, K, alpha, A, B, beta, C, stream);
}

phx_status phx_gemm_f16tc_f32acc(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                                 const float* B, float beta, float* C, phx_stream_t stream) {
    return gemm_entry(PHX_VARIANT_F16TC, M, N, K, alpha, A, B, beta, C, stream);
}

phx_status phx_sgemm_ex(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K, float alpha,
                        const float* A, const float* B, float beta, float* C, phx_stream_t stream) {
    if (!valid_op(op_a) || !valid_op(op_b)) return PHX_ERR_INVALID;
    return gemm_entry(PHX_VARIANT_SGEMM, M, N, K, alpha, A, B, beta, C, stream, op_a == PHX_OP_T,
                      op_b == PHX_OP_T);
}

phx_status phx_gemm_f16tc_f32acc_ex(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K,
                                    float alpha, const float* A, const float* B, float beta, float* C,
                                    phx_stream_t stream) {
    if (!valid_op(op_a) || !valid_op(op_b)) return PHX_ERR_INVALID;
    return gemm_entry(PHX_VARIANT_F16TC, M, N, K, alpha, A, B, beta, C, stream, op_a == PHX_OP_T,
                      op_b == PHX_OP_T);
}

phx_status phx_gemm_f16in_f32acc(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K, float alpha,
                                 const phx_f16* A, const phx_f16* B, float beta, float* C,
                                 phx_stream_t stream) {
    if (!valid_op(op_a) || !valid_op(op_b)) return PHX_ERR_INVALID;
    return f16in_entry(op_a == PHX_OP_T, op_b == PHX_OP_T, M, N, K, alpha, A, B, beta, C, nullptr, stream);
}

phx_status phx_gemm_f16in_f16out(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K, float alpha,
                                 const phx_f16* A, const phx_f16* B, float beta, phx_f16* C,
                                 phx_stream_t stream) {
    if (!valid_op(op_a) || !valid_op(op_b)) return PHX_ERR_INVALID;
    return f16in_entry(op_a == PHX_OP_T, op_b == PHX_OP_T, M, N, K, alpha, A, B, beta, nullptr,
                       reinterpret_cast<__half*>(C), stream);
}

phx_status phx_f16tc_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (bytes == nullptr || M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return PHX_ERR_INVALID;
    *bytes = phx::f16tc_workspace_bytes(M, N, K);
    return PHX_OK;
}

phx_status phx_check_device_status(phx_stream_t stream) {
    // Reads and clears both status words of the current device: the one of the pooled entry
    // points (if any of them ran here) and the one inside the allocation-free entry point's
    // static scratch (if that ran here).  Allocates nothing.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_ARCH;
    }
    unsigned int* pooled_word = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end() && it->second.ready) {
            if (it->second.init_status != PHX_OK) return it->second.init_status;
            pooled_word = it->second.status;
        }
    }
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_LAUNCH;
    }
    unsigned int word = 0;
    if (pooled_word != nullptr &&
        (cudaMemcpy(&word, pooled_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
         cudaMemset(pooled_word, 0, sizeof word) != cudaSuccess)) {
        cudaGetLastError();
        return PHX_ERR_LAUNCH;
    }
    unsigned int noalloc_word = 0;
    if (phx::noalloc_take_status(&noalloc_word) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_LAUNCH;
    }
    return ((word | noalloc_word) & phx::kDevTimeout) ? PHX_ERR_TIMEOUT : PHX_OK;
}

int phx_debug_build(void) {
#if defined(PHX_DEBUG) && PHX_DEBUG
    return 1;
#else
    return 0;
#endif
}

phx_status phx_debug_violations(int64_t* count) {
    if (count == nullptr) return PHX_ERR_INVALID;
    *count = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_ARCH;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_LAUNCH;
    }
    const int64_t parts[4] = {phx::debug_take_sgemm(), phx::debug_take_f16tc(), phx::debug_take_f16cvt(),
                              phx::debug_take_skinny()};
    for (int64_t v : parts) {
        if (v < 0) return PHX_ERR_LAUNCH;
        *count += v;
    }
    return PHX_OK;
}

phx_status phx_profile_start(void) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (auto& m : g_prof.marks) {
        g_prof.spare.push_back(std::get<1>(m));
        g_prof.spare.push_back(std::get<2>(m));
    }
    g_prof.marks.clear();
    g_prof.on = true;
    return PHX_OK;
}

phx_status phx_profile_stop(int64_t* launches, double* ms) {
    if (launches == nullptr || ms == nullptr) return PHX_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof.on = false;
    phx_status st = PHX_OK;
    for (int k = 0; k < kNumKinds; ++k) {
        launches[k] = 0;
        ms[k] = 0.0;
    }
    for (auto& m : g_prof.marks) {
        const int kind = std::get<0>(m);
        float t = 0.f;
        if (cudaEventSynchronize(std::get<2>(m)) != cudaSuccess ||
            cudaEventElapsedTime(&t, std::get<1>(m), std::get<2>(m)) != cudaSuccess) {
            cudaGetLastError();
            st = PHX_ERR_LAUNCH;
        }
        launches[kind] += std::get<3>(m);
        ms[kind] += t;
        g_prof.spare.push_back(std::get<1>(m));
        g_prof.spare.push_back(std::get<2>(m));
    }
    g_prof.marks.clear();
    return st;
}

int phx_num_configs(int variant) { return num_configs(variant); }

phx_status phx_config_name(int variant, int index, char* buf, size_t buflen) {
    const int n = num_configs(variant);
    if (n < 0 || index < 0 || index >= n) return PHX_ERR_INVALID;
    return copy_name(config_name(variant, index), buf, buflen);
}

phx_status phx_set_config(int variant, const char* spec) {
    if (num_configs(variant) < 0) return PHX_ERR_INVALID;
    int idx = -1;
    if (spec != nullptr && spec[0] != '\0') {
        idx = parse_config(variant, spec);
        if (idx < 0) return PHX_ERR_CONFIG;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    load_env_once_locked();
    g_pin[variant] = idx;
    return PHX_OK;
}

phx_status phx_get_config(int variant, int64_t M, int64_t N, int64_t K, char* buf, size_t buflen) {
    if (num_configs(variant) < 0 || M < 0 || N < 0 || K < 0) return PHX_ERR_INVALID;
    int sms = 148;
    DevState* d = nullptr;
    if (device_state(&d) == PHX_OK) sms = d->sm_count;
    const int cfg = choose_config(variant, M, N, K, sms);
    if (cfg < 0) return config_error(cfg);
    return copy_name(config_name(variant, cfg), buf, buflen);
}

phx_status phx_last_config(int variant, char* buf, size_t buflen) {
    if (num_configs(variant) < 0) return PHX_ERR_INVALID;
    const int cfg = g_last_cfg[variant].load();
    return copy_name(cfg < 0 ? std::string("NONE") : config_name(variant, cfg), buf, buflen);
}

phx_status phx_autotune(int variant, int64_t M, int64_t N, int64_t K, int finalists, int rounds,
                        int settle_ms, phx_stream_t stream) {
    const int n = num_configs(variant);
    if (n < 0 || M <= 0 || N <= 0 || K <= 0) return PHX_ERR_INVALID;
    if (validate_sizes(M, N, K) != PHX_OK) return PHX_ERR_INVALID;
    DevState* d = nullptr;
    phx_status st = device_state(&d);
    if (st != PHX_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    const std::string tag = device_tag();
    float *A = nullptr, *B = nullptr, *C = nullptr;
    if (cudaMalloc(&A, 4 * M * K) != cudaSuccess || cudaMalloc(&B, 4 * K * N) != cudaSuccess ||
        cudaMalloc(&C, 4 * M * N) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(A); cudaFree(B); cudaFree(C);
        return PHX_ERR_NOMEM;
    }
    tune_fill_kernel<<<1024, 256, 0, stream>>>(A, M * K, 0x1234u);
    tune_fill_kernel<<<1024, 256, 0, stream>>>(B, K * N, 0x5678u);
    tune_fill_kernel<<<1024, 256, 0, stream>>>(C, M * N, 0x9abcu);
    const char* inject = std::getenv("PHX_TUNE_FAIL");  // fault injection: this config "fails"
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    auto measure = [&](int i) -> double {
        if (inject != nullptr && config_name(variant, i) == inject) return -1.0;
        cudaEventRecord(e0, stream);
        const phx_status s = launch_variant(variant, i, M, N, K, 1.0f, A, B, 0.5f, C, d, stream);
        cudaEventRecord(e1, stream);
        if (s != PHX_OK || cudaEventSynchronize(e1) != cudaSuccess) {
            cudaGetLastError();
            return -1.0;
        }
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        return ms * 1e-3;
    };
    const auto start = std::chrono::steady_clock::now();
    auto elapsed = [&]() {
        return std::chrono::duration<double>(std::chrono::steady_clock::now() - start).count();
    };
    // every second-stage timing with the SM clock read right after it (NVML, -1 if absent)
    std::map<int, std::vector<std::pair<double, double>>> stage2;
    auto stage2_timed = [&](int i, double sec) { stage2[i].emplace_back(sec, sm_clock_mhz(dev)); };
    const TuneOutcome res = tune_select(n, measure, elapsed, finalists > 0 ? finalists : 4,
                                        rounds > 0 ? rounds : 9, settle_ms > 0 ? settle_ms * 1e-3 : 0.25,
                                        0x5eedull ^ static_cast<uint64_t>(M * 31 + N * 17 + K), stage2_timed);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaStreamSynchronize(stream);
    cudaFree(A);
    cudaFree(B);
    cudaFree(C);
    // A timeout during tuning is reported, not hidden.
    st = phx_check_device_status(stream);
    if (st != PHX_OK) return st;
    if (res.picked < 0) return PHX_ERR_LAUNCH;
    // The report of this run: one line per finalist with its median time and the median SM
    // clock of its timings.
    std::ostringstream rep;
    rep << "device " << tag << " variant " << variant << " shape " << M << ' ' << N << ' ' << K
        << " picked " << config_name(variant, res.picked) << " launches " << res.launches << '\n';
    for (const auto& kv : stage2) {
        std::vector<double> t, c;
        for (const auto& x : kv.second) {
            t.push_back(x.first);
            if (x.second > 0) c.push_back(x.second);
        }
        char line[256];
        std::snprintf(line, sizeof line, "  %-48s median_ms %.4f sm_mhz %.0f timings %zu\n",
                      config_name(variant, kv.first).c_str(), 1e3 * median(t), c.empty() ? -1.0 : median(c),
                      t.size());
        rep << line;
    }
    if (log_level() >= 1) std::fprintf(stderr, "[phx] tuned: %s", rep.str().c_str());
    std::lock_guard<std::mutex> lock(g_mu);
    g_tune_report[variant] = rep.str();
    g_tuned[ShapeKey(tag, variant, M, N, K)] = res.picked;
    if (const char* path = std::getenv("PHX_TUNE_CACHE")) {
        if (tune_cache_write_locked(path) != PHX_OK)
            std::fprintf(stderr, "[phx] PHX_TUNE_CACHE=%s could not be written\n", path);
    }
    return PHX_OK;
}

phx_status phx_autotune_report(int variant, char* buf, size_t buflen) {
    if (num_configs(variant) < 0) return PHX_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_mu);
    return copy_name(g_tune_report[variant].empty() ? std::string("NONE\n") : g_tune_report[variant], buf, buflen);
}

phx_status phx_device_tag(char* buf, size_t buflen) { return copy_name(device_tag(), buf, buflen); }

phx_status phx_tune_cache_save(const char* path) {
    if (path == nullptr) return PHX_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_mu);
    return tune_cache_write_locked(path);
}

phx_status phx_tune_cache_load(const char* path) {
    if (path == nullptr) return PHX_ERR_INVALID;
    std::map<ShapeKey, int> loaded;
    const phx_status st = tune_cache_read(path, &loaded);
    if (st != PHX_OK) return st;
    std::lock_guard<std::mutex> lock(g_mu);
    for (const auto& kv : loaded) g_tuned[kv.first] = kv.second;
    return PHX_OK;
}

phx_status phx_probe_ffma(int packed, int64_t blocks, int iters, float* out, phx_stream_t stream) {
    if (blocks <= 0 || blocks > 0x7FFFFFFF || iters <= 0 || out == nullptr) return PHX_ERR_INVALID;
    DevState* d = nullptr;
    phx_status st = device_state(&d);
    if (st != PHX_OK) return st;
    return phx::probe_ffma_launch(packed, blocks, iters, out, stream) == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

phx_status phx_probe_stream_read(const float* x, int64_t n, uint32_t* fold, int64_t blocks,
                                 phx_stream_t stream) {
    if (x == nullptr || fold == nullptr || n <= 0 || n % 4 != 0 || blocks <= 0 || blocks > 0x7FFFFFFF ||
        (reinterpret_cast<uintptr_t>(x) & 15u) != 0)
        return PHX_ERR_INVALID;
    DevState* d = nullptr;
    phx_status st = device_state(&d);
    if (st != PHX_OK) return st;
    return phx::probe_stream_read_launch(x, n, fold, blocks, stream) == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

phx_status phx_probe_mma_f16(int64_t ctas, int iters, int n, float* sink, phx_stream_t stream) {
    if (ctas <= 0 || ctas > 0x7FFFFFFF || iters <= 0 || sink == nullptr || (n != 64 && n != 128 && n != 256))
        return PHX_ERR_INVALID;
    DevState* d = nullptr;
    phx_status st = device_state(&d);
    if (st != PHX_OK) return st;
    return phx::probe_mma_f16_launch(ctas, iters, n, sink, d->status, stream) == cudaSuccess ? PHX_OK
                                                                                               : PHX_ERR_LAUNCH;
}

phx_status phx_selftest_bounded_wait(uint64_t limit_ns, phx_stream_t stream) {
    DevState* d = nullptr;
    phx_status st = device_state(&d);
    if (st != PHX_OK) return st;
    limit_ns = std::min<uint64_t>(std::max<uint64_t>(limit_ns, 1000), 1000000000ull);
    return phx::selftest_wait_launch(limit_ns, d->status, stream) == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
}

phx_status phx_selftest_sgemm_schedule(int config, int64_t M, int64_t N, int64_t K, int ctas_per_sm, int num_sms,
                                       int64_t* out) {
    if (out == nullptr || config < 0 || config >= phx::sgemm_num_configs() || ctas_per_sm <= 0 || ctas_per_sm > 32 ||
        num_sms <= 0 || num_sms > 4096 || M <= 0 || N <= 0 || K <= 0 || validate_sizes(M, N, K) != PHX_OK)
        return PHX_ERR_INVALID;
    phx::sgemm_schedule_selftest(config, M, N, K, ctas_per_sm, num_sms, out);
    return PHX_OK;
}

phx_status phx_selftest_tuner(int n, const double* base_s, const int* fail, double noise,
                              double drift, int finalists, int rounds, uint64_t seed, int* picked,
                              int64_t* launches) {
    if (n <= 0 || base_s == nullptr || picked == nullptr || launches == nullptr) return PHX_ERR_INVALID;
    double clock = 0.0;
    int64_t calls = 0;
    auto measure = [&](int i) -> double {
        ++calls;
        if (fail != nullptr && fail[i]) return -1.0;
        // deterministic noise in [-1, 1) from a hash of (seed, call)
        uint64_t h = (seed + static_cast<uint64_t>(calls)) * 0x9E3779B97F4A7C15ull;
        h ^= h >> 31;
        h *= 0xBF58476D1CE4E5B9ull;
        h ^= h >> 29;
        const double u = static_cast<double>(h >> 11) * (1.0 / 9007199254740992.0) * 2.0 - 1.0;
        const double s = base_s[i] * (1.0 + drift * static_cast<double>(calls)) * (1.0 + noise * u);
        clock += s;
        return s;
    };
    auto elapsed = [&]() { return clock; };
    const double total = std::accumulate(base_s, base_s + n, 0.0);
    const TuneOutcome res = tune_select(n, measure, elapsed, finalists, rounds, 2.0 * total, seed);
    *picked = res.picked;
    *launches = res.launches;
    return PHX_OK;
}

}  // extern "C"

namespace phx {

void note_launches(int n) { t_launches += n; }

cudaError_t set_func_attr_once(const void* fn, cudaFuncAttribute attr, int value) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, int>, bool> done;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const auto key = std::make_tuple(dev, fn, static_cast<int>(attr), value);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (done.count(key)) return cudaSuccess;
    }
    err = cudaFuncSetAttribute(fn, attr, value);
    if (err == cudaSuccess) {
        std::lock_guard<std::mutex> lock(mu);
        done[key] = true;
    }
    return err;
}

int64_t noted_launches() { return t_launches; }

}  // namespace phx
