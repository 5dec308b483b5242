// The C ABI of include/mica_optim.h: host-side validation, the per-list device tables (cached), the step's scalars,
// and the launches. Nothing here touches tensor data; every element is read and written by the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "host.h"
#include "mica_optim.h"
#include "plan.h"

namespace mica {

// ------------------------------------------------------------------------------------------------------------------
// bookkeeping: launch count, per-thread error detail, debug synchronisation
// ------------------------------------------------------------------------------------------------------------------

static std::atomic<uint64_t> g_launches{0};
void count_launches(uint64_t k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

static thread_local std::string t_detail;

void set_error_detail(const char* msg) { t_detail = msg; }

static mica_status fail(mica_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_detail = buf;
    return s;
}

static mica_status ok() {
    t_detail.clear();
    return MICA_OK;
}

static mica_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MICA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

static bool sync_debug() {
    static const bool on = [] {
        const char* s = std::getenv("MICA_SYNC_DEBUG");
        return s && s[0] && std::strcmp(s, "0") != 0;
    }();
    return on;
}

// After a stream has drained: a kernel whose bounded pipeline wait gave up leaves a nonzero device status word.
static mica_status check_device_status(const char* what) {
    unsigned int st = 0, fst = 0;
    int e = read_device_status(&st);
    if (e == (int)cudaSuccess) e = read_fused_status(&fst);
    if (e != (int)cudaSuccess) return cuda_fail((cudaError_t)e, what);
    if (fst) return fail(MICA_ERR_CUDA, "%s: a fused kernel's grid-wide wait gave up (status 0x%x); its results are "
                         "not valid, and the list's table must be released (mica_release_cache)", what, fst);
    if (st) return fail(MICA_ERR_CUDA, "%s: a kernel's wait on its shared-memory pipeline gave up (status 0x%x); "
                        "its results are not valid", what, st);
    return MICA_OK;
}

static mica_status after_launch(int err, void* stream, const char* what) {
    if (err != (int)cudaSuccess) return cuda_fail((cudaError_t)err, what);
    if (sync_debug()) {
        const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, what);
        const mica_status s = check_device_status(what);
        if (s != MICA_OK) return s;
    }
    return ok();
}

// ------------------------------------------------------------------------------------------------------------------
// pointer checks (only when a list's table is built, and for the scalar outputs of each call)
// ------------------------------------------------------------------------------------------------------------------

using MemGetAddressRange = int (*)(unsigned long long* base, size_t* size, unsigned long long ptr);

static MemGetAddressRange address_range_fn() {
    static MemGetAddressRange fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (MemGetAddressRange) nullptr;
        }
        return reinterpret_cast<MemGetAddressRange>(p);
    }();
    return fn;
}

mica_status check_device_span(const void* p, size_t bytes, size_t align, int device, const char* what,
                                     int64_t index) {
    if (reinterpret_cast<uintptr_t>(p) % align != 0)
        return fail(MICA_ERR_ADDRESS, "%s[%lld] = %p is not %zu-byte aligned", what, (long long)index, p, align);
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(MICA_ERR_ADDRESS, "%s[%lld] = %p: cudaPointerGetAttributes failed (%s)", what, (long long)index,
                    p, cudaGetErrorName(e));
    }
    if (a.type == cudaMemoryTypeDevice) {
        if (a.device != device)
            return fail(MICA_ERR_ADDRESS, "%s[%lld] = %p is memory of device %d, not of the current device %d", what,
                        (long long)index, p, a.device, device);
    } else if (a.type != cudaMemoryTypeManaged) {
        return fail(MICA_ERR_ADDRESS, "%s[%lld] = %p is not device memory", what, (long long)index, p);
    }
    if (MemGetAddressRange fn = address_range_fn()) {
        unsigned long long base = 0;
        size_t size = 0;
        if (fn(&base, &size, (unsigned long long)reinterpret_cast<uintptr_t>(p)) == 0) {
            const unsigned long long end = base + size, q = (unsigned long long)reinterpret_cast<uintptr_t>(p);
            if (q + bytes > end)
                return fail(MICA_ERR_ADDRESS, "%s[%lld] = %p: %zu bytes run past the end of its allocation", what,
                            (long long)index, p, bytes);
        }
    }
    return MICA_OK;
}

struct Span {
    uintptr_t lo, hi;  // [lo, hi)
    int32_t kind, index;
};

static const char* span_name(int32_t kind) {
    static const char* names[] = {"w", "g", "m", "v", "t", "buf", "a"};
    return names[kind];
}

// sorts `spans` and fails when two overlap
static mica_status check_disjoint(std::vector<Span>& spans) {
    std::sort(spans.begin(), spans.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
    for (size_t i = 1; i < spans.size(); ++i)
        if (spans[i].lo < spans[i - 1].hi)
            return fail(MICA_ERR_OVERLAP, "%s[%d] overlaps %s[%d]", span_name(spans[i].kind), spans[i].index,
                        span_name(spans[i - 1].kind), spans[i - 1].index);
    return MICA_OK;
}

static bool overlaps_any(const std::vector<Span>& sorted, const void* p, size_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p), hi = lo + bytes;
    auto it = std::upper_bound(sorted.begin(), sorted.end(), lo, [](uintptr_t x, const Span& s) { return x < s.lo; });
    if (it != sorted.end() && it->lo < hi) return true;
    if (it != sorted.begin() && std::prev(it)->hi > lo) return true;
    return false;
}

// ------------------------------------------------------------------------------------------------------------------
// per-list device tables
// ------------------------------------------------------------------------------------------------------------------

enum Kind : uint64_t { kAdamW = 1, kNorm = 2, kScale = 3, kSGD = 4, kMomentum = 5, kAccNorm = 6 };

struct Plan {
    // the list it was built for (compared in full on every lookup)
    Kind kind = kAdamW;
    int device = 0;
    Dtype gdt = kF32, mdt = kF32;
    int32_t T = 0;
    std::vector<int64_t> n;
    std::vector<const void*> ptrs[4];  // the pointer arrays the kind uses, in ListDesc order
    std::vector<int32_t> group;        // AdamW over parameter groups: each tensor's group (empty: none)
    int32_t max_group = 0;             // the largest entry of `group`
    int64_t total = 0;                 // elements
    const void* checked_scalar[2] = {nullptr, nullptr};  // the last scalar outputs found valid for this list
    void* dev = nullptr;  // one allocation: TensorRec[T] | WorkItem[I] | pack table | the norm's tables
    TensorRec* recs = nullptr;
    WorkItem* items = nullptr;
    int32_t* pack_pre = nullptr;  // per pack: the first pack octet of each tensor, and the total
    unsigned int* queues = nullptr;  // kQueues work queues of the update kernels' persistent grids (2 counters each)
    std::atomic<uint32_t> launches{0};  // update launches so far: launch i uses queue i % kQueues
    int32_t sms = 0;
    int32_t num_items = 0;
    int32_t item_octs = 0;
    // norm plans
    ChunkTable chunks{};
    double* partials = nullptr;
    unsigned int* ticket = nullptr;  // the finishing-order counter of the fused finalize
    std::vector<Span> spans;  // the list's buffers, sorted (for checking a call's scalar outputs)
    // AdamW plans used by mica_clip_adamw_step: the gradient in equal chunks, one per CTA of the fused launch
    // (records, octet prefix, chunk starts), the per-CTA partials and the grid-wide wait's two words; built on the
    // first fused call, in an allocation of its own
    void* fdev = nullptr;
    ChunkTable fchunks{};
    double* fpartials = nullptr;
    unsigned int* fbar = nullptr;
    int32_t pins = 0;  // calls in progress that hold this table (under g_mu; see CallScope)
    ~Plan() {
        if (dev || fdev) {
            int cur = 0;
            cudaGetDevice(&cur);
            cudaSetDevice(device);
            if (dev) cudaFree(dev);
            if (fdev) cudaFree(fdev);
            cudaSetDevice(cur);
        }
    }
};

// Work queues per list: a launch may overlap the one before it (programmatic dependent launch), never one of
// several launches before, so a handful of queues used in turn keeps overlapping launches apart.
constexpr int kQueues = 8;

static std::mutex g_mu;
static std::unordered_map<uint64_t, std::vector<std::unique_ptr<Plan>>> g_plans;
static size_t g_plan_count = 0;
constexpr size_t kMaxPlans = 1024;

// Tables a call in progress holds. Every table a call looks up is pinned until the outermost library call of its
// thread returns (each entry point opens a CallScope), and neither the cache's eviction nor mica_release_cache frees
// a pinned table: so a call that looks up a second list after its first (mica_clip_adamw_step's norm) never loses
// the first, and calls in progress on other threads keep theirs.
static thread_local int t_call_depth = 0;
static thread_local std::vector<Plan*> t_pinned;

struct CallScope {
    CallScope() { ++t_call_depth; }
    ~CallScope() {
        if (--t_call_depth == 0 && !t_pinned.empty()) {
            std::lock_guard<std::mutex> lock(g_mu);
            for (Plan* p : t_pinned) --p->pins;
            t_pinned.clear();
        }
    }
    CallScope(const CallScope&) = delete;
    CallScope& operator=(const CallScope&) = delete;
};

// Pins a table for the calling thread's outermost call (g_mu held).
static void pin_plan(Plan* p) {
    if (p && t_call_depth > 0) {
        ++p->pins;
        t_pinned.push_back(p);
    }
}

// Frees every cached table that no call in progress holds (g_mu held; the device is idle).
static void evict_unpinned() {
    size_t kept = 0;
    for (auto it = g_plans.begin(); it != g_plans.end();) {
        auto& v = it->second;
        v.erase(std::remove_if(v.begin(), v.end(), [](const std::unique_ptr<Plan>& p) { return p->pins == 0; }),
                v.end());
        kept += v.size();
        it = v.empty() ? g_plans.erase(it) : std::next(it);
    }
    g_plan_count = kept;
}

static uint64_t mix(uint64_t h, uint64_t x) {
    h ^= x + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
    return h * 0xFF51AFD7ED558CCDull;
}

static int sm_count(int device) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 148;
    }
    return n;
}

// Octets per slice of a large tensor, measured best on GB300 for each kernel and stream set (the update kernels run
// as persistent grids): AdamW with float32 moments 512 (4,096 elements: 64 KB of loads), AdamW with packed moments
// 1024, SGD 1024, SGD with momentum 512, ScaleTensors 2048; halved down to 128 for small lists so that all SMs still
// get work. MICA_ITEM_OCTS overrides it (a power of two).
static int32_t base_item_octs(Kind kind, Dtype mdt) {
    if (kind == kAdamW) return mdt == kF32 ? 512 : 1024;
    if (kind == kMomentum) return 512;
    if (kind == kSGD) return 1024;
    return 2048;
}

static int32_t choose_item_octs(int64_t total_octs, int sms, int32_t base) {
    if (const char* s = std::getenv("MICA_ITEM_OCTS")) {
        const long v = std::strtol(s, nullptr, 10);
        if (v >= 16 && v <= (1 << 20) && (v & (v - 1)) == 0) return (int32_t)v;
    }
    int32_t io = base;
    const int64_t target = (int64_t)sms * 16;
    while (io > 128 && total_octs / io < target) io /= 2;
    return io;
}

// Work items over the tensors' octets (see plan.h), and the pack table. A pack of two or more tensors numbers its
// octets whole octets of aligned tensors first (tensor by tensor), then the rest (each aligned tensor's partial last
// octet, every octet of an unaligned tensor), so that the element-by-element octets share warps with each other and
// not with the vector ones; its row of the pack table (from its item's o0) is the first whole octet of each tensor
// and the whole octets' total, then the first of each tensor's other octets and their total (2 count + 2 entries).
// Tensors of up to 512 octets (and at most io) are packed, up to 1536 octets a pack (and at most 3 io): measured
// best on GB300 for lists of thousands of small tensors.
static std::vector<WorkItem> build_items(const int64_t* n, const TensorRec* recs, int32_t T, int32_t io,
                                         std::vector<int32_t>* pack_pre) {
    std::vector<WorkItem> items;
    const int64_t small = std::min<int64_t>(512, io);
    const int64_t pack_cap = std::min<int64_t>(1536, 3 * (int64_t)io);
    bool open = false;
    WorkItem pack{};
    int64_t pack_o = 0;
    auto close = [&] {
        if (!open) return;
        if (pack.count > 1) {
            pack.o0 = (int64_t)pack_pre->size();
            auto whole = [&](int32_t k) { return recs[k].vec ? n[k] / kOct : (int64_t)0; };
            int32_t at = 0;
            for (int32_t j = 0; j < pack.count; ++j) {
                pack_pre->push_back(at);
                at += (int32_t)whole(pack.t + j);
            }
            pack_pre->push_back(at);
            at = 0;
            for (int32_t j = 0; j < pack.count; ++j) {
                pack_pre->push_back(at);
                at += (int32_t)((n[pack.t + j] + kOct - 1) / kOct - whole(pack.t + j));
            }
            pack_pre->push_back(at);
        }
        items.push_back(pack);
        open = false;
    };
    for (int32_t k = 0; k < T; ++k) {
        const int64_t no = (n[k] + kOct - 1) / kOct;
        if (no == 0) {
            if (open) pack.count += 1;  // an empty tensor inside a pack costs nothing
            continue;
        }
        if (no <= small) {
            if (open && pack_o + no <= pack_cap) {
                pack.count += 1;
                pack_o += no;
            } else {
                close();
                pack = WorkItem{k, 1, 0};
                pack_o = no;
                open = true;
            }
            continue;
        }
        close();
        for (int64_t o = 0; o < no; o += io) items.push_back(WorkItem{k, 1, o});
    }
    close();
    return items;
}

// The order the update kernels take the items in (they walk the array from its end): the packs first, spread
// evenly over as many slices as there are packs, then the other slices. A pack's CTA waits on memory latency far
// more than a slice's does (its threads' octets lie in many small tensors), so the packs run while slice CTAs keep
// HBM busy, and the launch ends on slices, its shortest and most even items, rather than on a wave of packs. Each
// kind keeps its own order (slices from the end of the list first).
static void order_items(std::vector<WorkItem>& items) {
    const size_t N = items.size();
    std::vector<WorkItem> S, P;  // in the order they are taken
    for (size_t j = 0; j < N; ++j) {
        const WorkItem& it = items[N - 1 - j];
        (it.count > 1 ? P : S).push_back(it);
    }
    if (P.empty() || S.empty()) return;
    const int64_t np = (int64_t)P.size();
    const int64_t head = std::min<int64_t>((int64_t)S.size(), np);  // slices the packs are spread over
    std::vector<WorkItem> order;
    order.reserve(N);
    int64_t is = 0, ip = 0;
    while (is < head || ip < np) {
        if (ip < np && (is >= head || ip * head <= is * np)) order.push_back(P[(size_t)ip++]);
        else order.push_back(S[(size_t)is++]);
    }
    while ((size_t)is < S.size()) order.push_back(S[(size_t)is++]);
    for (size_t j = 0; j < N; ++j) items[N - 1 - j] = order[j];
}

static uint64_t ptr_u(const void* p) { return (uint64_t) reinterpret_cast<uintptr_t>(p); }

struct ListDesc {
    Kind kind;
    int32_t T;
    const int64_t* n;
    float* const* w;     // adamw: weights; scale: the tensors
    void* const* g;      // adamw, norm
    void* const* m;      // adamw; accumulate: the addends
    void* const* v;      // adamw
    Dtype gdt, mdt;      // scale: gdt is the tensors' type
    const int32_t* group = nullptr;  // AdamW over parameter groups: T group indices (validated by the caller)
};

static size_t elem_bytes(Dtype d) { return d == kF16 ? 2 : 4; }

static int list_arrays(const ListDesc& L, const void* const* out[4]) {
    if (L.kind == kScale) {
        out[0] = reinterpret_cast<const void* const*>(L.w);
        return 1;
    }
    if (L.kind == kNorm) {
        out[0] = L.g;
        return 1;
    }
    if (L.kind == kAccNorm) {
        out[0] = L.g;
        out[1] = L.m;  // the addends
        return 2;
    }
    if (L.kind == kSGD || L.kind == kMomentum) {
        out[0] = reinterpret_cast<const void* const*>(L.w);
        out[1] = L.g;
        out[2] = L.m;  // the momentum buffers
        return L.kind == kMomentum ? 3 : 2;
    }
    out[0] = reinterpret_cast<const void* const*>(L.w);
    out[1] = L.g;
    out[2] = L.m;
    out[3] = L.v;
    return 4;
}

// A hash of the list from its header and a sample of its entries (at most ~64): cheap for lists of any length.
// Lookups compare the whole list, so a shared hash only costs a comparison.
static uint64_t list_hash(const ListDesc& L, int device) {
    uint64_t h = 0x243F6A8885A308D3ull;
    h = mix(h, (uint64_t)L.kind);
    h = mix(h, (uint64_t)device);
    h = mix(h, ((uint64_t)L.gdt << 8) | (uint64_t)L.mdt);
    h = mix(h, (uint64_t)L.T);
    h = mix(h, L.group ? 1u : 0u);
    if (L.T == 0) return h;
    const void* const* arr[4];
    const int na = list_arrays(L, arr);
    const int32_t step = L.T > 64 ? L.T / 64 : 1;
    for (int32_t k = 0; k < L.T; k += step) {
        h = mix(h, (uint64_t)L.n[k]);
        for (int a = 0; a < na; ++a) h = mix(h, ptr_u(arr[a][k]));
        if (L.group) h = mix(h, (uint64_t)(uint32_t)L.group[k]);
    }
    h = mix(h, (uint64_t)L.n[L.T - 1]);
    for (int a = 0; a < na; ++a) h = mix(h, ptr_u(arr[a][L.T - 1]));
    return h;
}

static bool same_list(const Plan& p, const ListDesc& L, int device) {
    if (p.kind != L.kind || p.device != device || p.gdt != L.gdt || p.mdt != L.mdt || p.T != L.T) return false;
    if (L.T == 0) return true;
    if (std::memcmp(p.n.data(), L.n, (size_t)L.T * sizeof(int64_t)) != 0) return false;
    const void* const* arr[4];
    const int na = list_arrays(L, arr);
    for (int a = 0; a < na; ++a)
        if (std::memcmp(p.ptrs[a].data(), arr[a], (size_t)L.T * sizeof(void*)) != 0) return false;
    if (p.group.empty() != (L.group == nullptr)) return false;
    if (L.group && std::memcmp(p.group.data(), L.group, (size_t)L.T * sizeof(int32_t)) != 0) return false;
    return true;
}

static mica_status build_plan(const ListDesc& L, int device, uint64_t h, Plan** out, void* stream) {
    auto plan = std::make_unique<Plan>();
    plan->kind = L.kind;
    plan->device = device;
    plan->gdt = L.gdt;
    plan->mdt = L.mdt;
    plan->T = L.T;
    if (L.T > 0) {
        plan->n.assign(L.n, L.n + L.T);
        const void* const* arr[4];
        const int na = list_arrays(L, arr);
        for (int a = 0; a < na; ++a) plan->ptrs[a].assign(arr[a], arr[a] + L.T);
        if (L.group) {
            plan->group.assign(L.group, L.group + L.T);
            plan->max_group = *std::max_element(plan->group.begin(), plan->group.end());
        }
    }
    for (int32_t k = 0; k < L.T; ++k) plan->total += L.n[k];

    // pointer checks and the overlap check, over every non-empty buffer of the list
    std::vector<Span> spans;
    std::vector<TensorRec> recs((size_t)L.T);
    int64_t total_octs = 0;
    for (int32_t k = 0; k < L.T; ++k) {
        const int64_t n = L.n[k];
        TensorRec& r = recs[k];
        r = TensorRec{nullptr, nullptr, nullptr, nullptr, n, 0, L.group ? L.group[k] : 0};
        if (n == 0) continue;
        total_octs += (n + kOct - 1) / kOct;
        mica_status s;
        if (L.kind == kScale) {
            const size_t b = (size_t)n * elem_bytes(L.gdt);
            if ((s = check_device_span(L.w[k], b, elem_bytes(L.gdt), device, "t", k)) != MICA_OK) return s;
            r.w = L.w[k];
            r.vec = (ptr_u(r.w) % (L.gdt == kF16 ? 16 : 32)) == 0;
            spans.push_back({(uintptr_t)ptr_u(r.w), (uintptr_t)(ptr_u(r.w) + b), 4, k});
            continue;
        }
        const size_t gb = (size_t)n * elem_bytes(L.gdt);
        if ((s = check_device_span(L.g[k], gb, elem_bytes(L.gdt), device, "g", k)) != MICA_OK) return s;
        r.g = L.g[k];
        spans.push_back({(uintptr_t)ptr_u(r.g), (uintptr_t)(ptr_u(r.g) + gb), 1, k});
        bool vec = (ptr_u(r.g) % (L.gdt == kF16 ? 16 : 32)) == 0;
        if (L.kind == kAccNorm) {
            if ((s = check_device_span(L.m[k], gb, elem_bytes(L.gdt), device, "a", k)) != MICA_OK) return s;
            r.m = L.m[k];
            spans.push_back({(uintptr_t)ptr_u(r.m), (uintptr_t)(ptr_u(r.m) + gb), 6, k});
            vec = vec && (ptr_u(r.m) % (L.gdt == kF16 ? 16 : 32)) == 0;
        } else if (L.kind == kAdamW) {
            const size_t wb = (size_t)n * 4;
            const size_t packed_b = (size_t)((n + 1) / 2) * 4, f32_b = (size_t)n * 4;
            const size_t mb = (L.mdt == kBF16x2 || L.mdt == kBF16x2M) ? packed_b : f32_b;
            const size_t vb = (L.mdt == kBF16x2) ? packed_b : f32_b;
            if ((s = check_device_span(L.w[k], wb, 4, device, "w", k)) != MICA_OK) return s;
            if ((s = check_device_span(L.m[k], mb, 4, device, "m", k)) != MICA_OK) return s;
            if ((s = check_device_span(L.v[k], vb, 4, device, "v", k)) != MICA_OK) return s;
            r.w = L.w[k];
            r.m = L.m[k];
            r.v = L.v[k];
            spans.push_back({(uintptr_t)ptr_u(r.w), (uintptr_t)(ptr_u(r.w) + wb), 0, k});
            spans.push_back({(uintptr_t)ptr_u(r.m), (uintptr_t)(ptr_u(r.m) + mb), 2, k});
            spans.push_back({(uintptr_t)ptr_u(r.v), (uintptr_t)(ptr_u(r.v) + vb), 3, k});
            const uint64_t ma = (L.mdt == kBF16x2 || L.mdt == kBF16x2M) ? 16 : 32;  // packed: 4 words an octet
            const uint64_t va = (L.mdt == kBF16x2) ? 16 : 32;
            vec = vec && ptr_u(r.w) % 32 == 0 && ptr_u(r.m) % ma == 0 && ptr_u(r.v) % va == 0;
        } else if (L.kind == kSGD || L.kind == kMomentum) {
            const size_t wb = (size_t)n * 4;
            if ((s = check_device_span(L.w[k], wb, 4, device, "w", k)) != MICA_OK) return s;
            r.w = L.w[k];
            spans.push_back({(uintptr_t)ptr_u(r.w), (uintptr_t)(ptr_u(r.w) + wb), 0, k});
            vec = vec && ptr_u(r.w) % 32 == 0;
            if (L.kind == kMomentum) {
                if ((s = check_device_span(L.m[k], wb, 4, device, "buf", k)) != MICA_OK) return s;
                r.m = L.m[k];
                spans.push_back({(uintptr_t)ptr_u(r.m), (uintptr_t)(ptr_u(r.m) + wb), 5, k});
                vec = vec && ptr_u(r.m) % 32 == 0;
            }
        }
        r.vec = vec ? 1 : 0;
    }
    if (L.kind != kNorm) {
        mica_status s = check_disjoint(spans);
        if (s != MICA_OK) return s;
    } else {
        std::sort(spans.begin(), spans.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
    }
    plan->spans = std::move(spans);

    const int sms = sm_count(device);
    std::vector<WorkItem> items;
    std::vector<int32_t> pack_pre;
    std::vector<int64_t> prefix;
    std::vector<int32_t> first;
    int64_t nonempty = 0;
    for (int32_t k = 0; k < L.T; ++k) nonempty += L.n[k] > 0;
    const bool chunked = L.kind == kNorm || L.kind == kAccNorm;
    if (chunked) {
        // contiguous equal chunks (see choose_norm_shape; the accumulating norm: the register-streaming layout)
        prefix.resize((size_t)L.T + 1);
        prefix[0] = 0;
        for (int32_t k = 0; k < L.T; ++k) prefix[k + 1] = prefix[k] + (L.n[k] + kOct - 1) / kOct;
        int32_t grid = 1, direct = 1;
        if (L.kind == kNorm)
            choose_norm_shape(total_octs, nonempty, L.gdt == kF16 ? 16 : 32, sms, INT32_MAX, &grid, &direct);
        else
            grid = choose_accumulate_grid(total_octs, L.gdt == kF16 ? 16 : 32, sms);
        plan->chunks.direct = direct;
        first.resize((size_t)grid);
        for (int32_t b = 0; b < grid; ++b) {
            const int64_t c0 = total_octs * b / grid;
            // the last tensor whose range starts at or before c0 (empty tensors share their start with the next)
            int32_t k = (int32_t)(std::upper_bound(prefix.begin(), prefix.end(), c0) - prefix.begin()) - 1;
            first[b] = std::max(0, std::min(k, std::max(0, L.T - 1)));
        }
        plan->chunks.T = L.T;
        plan->chunks.grid = grid;
        plan->chunks.total_octs = total_octs;
    } else {
        plan->item_octs = choose_item_octs(total_octs, sms, base_item_octs(L.kind, L.mdt));
        items = build_items(L.n, recs.data(), L.T, plan->item_octs, &pack_pre);
        order_items(items);
        if (items.size() > (size_t)INT32_MAX) return fail(MICA_ERR_COUNT, "too many work items (%zu)", items.size());
        plan->num_items = (int32_t)items.size();
    }

    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rec_b = recs.size() * sizeof(TensorRec);
    const size_t item_off = up(rec_b);
    const size_t item_b = items.size() * sizeof(WorkItem);
    const size_t pack_off = up(item_off + item_b);
    const size_t pack_b = pack_pre.size() * sizeof(int32_t);
    const size_t prefix_off = up(pack_off + pack_b);
    const size_t prefix_b = prefix.size() * sizeof(int64_t);
    const size_t first_off = up(prefix_off + prefix_b);
    const size_t first_b = first.size() * sizeof(int32_t);
    const size_t part_off = up(first_off + first_b);
    const size_t part_b = chunked ? first.size() * sizeof(double) : 0;
    const size_t ticket_off = up(part_off + part_b);
    const size_t ticket_b = chunked ? 256 : 0;
    const size_t queue_off = up(ticket_off + ticket_b);
    const size_t queue_b = (chunked || L.kind == kScale) ? 0 : kQueues * 2 * sizeof(unsigned int);
    const size_t total = queue_off + queue_b;
    cudaError_t e = cudaMalloc(&plan->dev, std::max<size_t>(total, 256));
    if (e != cudaSuccess) {
        cudaGetLastError();
        plan->dev = nullptr;
        return fail(MICA_ERR_NOMEM, "cudaMalloc of a %zu-byte tensor-list table failed (%s)", total,
                    cudaGetErrorName(e));
    }
    char* base = static_cast<char*>(plan->dev);
    plan->recs = reinterpret_cast<TensorRec*>(base);
    plan->items = reinterpret_cast<WorkItem*>(base + item_off);
    plan->pack_pre = reinterpret_cast<int32_t*>(base + pack_off);
    if (chunked) {
        plan->chunks.recs = plan->recs;
        plan->chunks.prefix = reinterpret_cast<const int64_t*>(base + prefix_off);
        plan->chunks.first = reinterpret_cast<const int32_t*>(base + first_off);
    }
    if (chunked) {
        plan->partials = reinterpret_cast<double*>(base + part_off);
        plan->ticket = reinterpret_cast<unsigned int*>(base + ticket_off);
    }
    plan->sms = sms;
    if (queue_b) {
        plan->queues = reinterpret_cast<unsigned int*>(base + queue_off);
        if ((e = cudaMemsetAsync(plan->queues, 0, queue_b, static_cast<cudaStream_t>(stream))) != cudaSuccess)
            return cuda_fail(e, "clearing the work queues");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (plan->ticket && (e = cudaMemsetAsync(plan->ticket, 0, sizeof(unsigned int), st)) != cudaSuccess)
        return cuda_fail(e, "clearing the norm's ticket");
    if (rec_b && (e = cudaMemcpyAsync(plan->recs, recs.data(), rec_b, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return cuda_fail(e, "uploading the tensor records");
    if (item_b && (e = cudaMemcpyAsync(plan->items, items.data(), item_b, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return cuda_fail(e, "uploading the work items");
    if (pack_b && (e = cudaMemcpyAsync(plan->pack_pre, pack_pre.data(), pack_b, cudaMemcpyHostToDevice, st)) !=
                      cudaSuccess)
        return cuda_fail(e, "uploading the pack table");
    if (prefix_b && (e = cudaMemcpyAsync(base + prefix_off, prefix.data(), prefix_b, cudaMemcpyHostToDevice, st)) !=
                        cudaSuccess)
        return cuda_fail(e, "uploading the octet prefix");
    if (first_b && (e = cudaMemcpyAsync(base + first_off, first.data(), first_b, cudaMemcpyHostToDevice, st)) !=
                       cudaSuccess)
        return cuda_fail(e, "uploading the chunk starts");
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "waiting for the table upload");
    *out = plan.get();

    if (g_plan_count >= kMaxPlans) {
        cudaDeviceSynchronize();
        evict_unpinned();
    }
    g_plans[h].push_back(std::move(plan));
    ++g_plan_count;
    return MICA_OK;
}

// The fused launch's norm table of an AdamW plan (see Plan::fdev), built once: grid = kFusedCtasPerSm CTAs per SM,
// CTA b summing octets [total*b/grid, total*(b+1)/grid) of the gradient, which starts in tensor first[b].
static mica_status ensure_fused_table(Plan* p, void* stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (p->fdev) return MICA_OK;
    const int32_t T = p->T;
    std::vector<TensorRec> recs((size_t)T);
    std::vector<int64_t> prefix((size_t)T + 1, 0);
    for (int32_t k = 0; k < T; ++k) {
        const int64_t n = p->n[k];
        const void* gp = n > 0 ? p->ptrs[1][k] : nullptr;
        recs[k] = TensorRec{nullptr, const_cast<void*>(gp), nullptr, nullptr, n, 0, 0};
        recs[k].vec = (ptr_u(gp) % (p->gdt == kF16 ? 16 : 32)) == 0;
        prefix[k + 1] = prefix[k] + (n + kOct - 1) / kOct;
    }
    const int64_t total_octs = prefix[T];
    const int32_t grid = kFusedCtasPerSm * p->sms;
    std::vector<int32_t> first((size_t)grid);
    for (int32_t b = 0; b < grid; ++b) {
        const int64_t c0 = total_octs * b / grid;
        int32_t k = (int32_t)(std::upper_bound(prefix.begin(), prefix.end(), c0) - prefix.begin()) - 1;
        first[b] = std::max(0, std::min(k, std::max(0, T - 1)));
    }
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rec_b = recs.size() * sizeof(TensorRec);
    const size_t prefix_off = up(rec_b), prefix_b = prefix.size() * sizeof(int64_t);
    const size_t first_off = up(prefix_off + prefix_b), first_b = first.size() * sizeof(int32_t);
    const size_t part_off = up(first_off + first_b), part_b = (size_t)grid * sizeof(double);
    const size_t bar_off = up(part_off + part_b), total = bar_off + 256;
    void* dev = nullptr;
    cudaError_t e = cudaMalloc(&dev, total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(MICA_ERR_NOMEM, "cudaMalloc of a %zu-byte fused norm table failed (%s)", total, cudaGetErrorName(e));
    }
    char* base = static_cast<char*>(dev);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rec_b && (e = cudaMemcpyAsync(base, recs.data(), rec_b, cudaMemcpyHostToDevice, st)) == cudaSuccess &&
        (e = cudaMemcpyAsync(base + prefix_off, prefix.data(), prefix_b, cudaMemcpyHostToDevice, st)) == cudaSuccess &&
        (e = cudaMemcpyAsync(base + first_off, first.data(), first_b, cudaMemcpyHostToDevice, st)) == cudaSuccess)
        e = cudaMemsetAsync(base + bar_off, 0, 256, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaFree(dev);
        return cuda_fail(e, "uploading the fused norm table");
    }
    p->fdev = dev;
    p->fchunks = ChunkTable{reinterpret_cast<const TensorRec*>(base), reinterpret_cast<const int64_t*>(base + prefix_off),
                            reinterpret_cast<const int32_t*>(base + first_off), T, grid, total_octs, 1, 0};
    p->fpartials = reinterpret_cast<double*>(base + part_off);
    p->fbar = reinterpret_cast<unsigned int*>(base + bar_off);
    return MICA_OK;
}

// The tables of one update launch on a cached list: a persistent grid with the next of the list's work queues, or
// (persistent false) one CTA per item. MICA_UPDATE_GRID=items / persistent overrides the choice unless `fixed`.
static UpdateLaunch update_launch(Plan* p, bool persistent, bool fixed = false) {
    if (const char* e = std::getenv("MICA_UPDATE_GRID"))
        if (!fixed) persistent = std::strcmp(e, "items") != 0;
    if (!persistent) return UpdateLaunch{p->recs, p->items, p->pack_pre, nullptr, p->num_items, p->item_octs, p->sms};
    const uint32_t i = p->launches.fetch_add(1, std::memory_order_relaxed) % kQueues;
    return UpdateLaunch{p->recs, p->items, p->pack_pre, p->queues + 2 * i, p->num_items, p->item_octs, p->sms};
}

// The cached table of a list, or nullptr.
static Plan* find_plan(const ListDesc& L, int device, uint64_t h) {
    auto it = g_plans.find(h);
    if (it == g_plans.end()) return nullptr;
    for (auto& p : it->second)
        if (same_list(*p, L, device)) return p.get();
    return nullptr;
}

// The table of an already validated list: the cached one, or a new one (which checks every pointer).
static mica_status get_plan(const ListDesc& L, int device, Plan** out, void* stream) {
    const uint64_t h = list_hash(L, device);
    std::lock_guard<std::mutex> lock(g_mu);
    mica_status s = MICA_OK;
    if ((*out = find_plan(L, device, h)) == nullptr) s = build_plan(L, device, h, out, stream);
    if (s == MICA_OK) pin_plan(*out);
    return s;
}

// A list seen before needs none of the per-tensor checks again: its counts and pointers equal those of a list that
// passed them when its table was built.
static Plan* cached_plan(const ListDesc& L, int device) {
    if (L.T <= 0) return nullptr;
    const uint64_t h = list_hash(L, device);
    std::lock_guard<std::mutex> lock(g_mu);
    Plan* p = find_plan(L, device, h);
    pin_plan(p);
    return p;
}

// The device scalars of a call (d_factor, d_norm): device memory of the current device, aligned, outside the list's
// buffers. The last pair found valid for a table is remembered, so a repeated call skips the driver queries.
static mica_status check_scalars(Plan* p, int dev, const float* a, const float* b, const char* what) {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (p->checked_scalar[0] == a && p->checked_scalar[1] == b) return MICA_OK;
    }
    const float* outs[2] = {a, b};
    const char* names[2] = {"d_factor", "d_norm"};
    for (int i = 0; i < 2; ++i) {
        if (!outs[i]) continue;
        mica_status s = check_device_span(outs[i], 4, 4, dev, names[i], 0);
        if (s != MICA_OK) return s;
        if (overlaps_any(p->spans, outs[i], 4)) return fail(MICA_ERR_OVERLAP, "%s lies inside %s", names[i], what);
    }
    if (a && b && reinterpret_cast<uintptr_t>(a) + 4 > reinterpret_cast<uintptr_t>(b) &&
        reinterpret_cast<uintptr_t>(b) + 4 > reinterpret_cast<uintptr_t>(a))
        return fail(MICA_ERR_OVERLAP, "d_norm and d_factor overlap");
    std::lock_guard<std::mutex> lock(g_mu);
    p->checked_scalar[0] = a;
    p->checked_scalar[1] = b;
    return MICA_OK;
}

// ------------------------------------------------------------------------------------------------------------------
// argument checks shared by the entry points
// ------------------------------------------------------------------------------------------------------------------

static mica_status check_list(int32_t T, const int64_t* n, std::initializer_list<const void* const*> arrays,
                              int64_t* total) {
    *total = 0;
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T == 0) return MICA_OK;
    if (!n) return fail(MICA_ERR_NULL, "the element-count array is NULL");
    for (auto a : arrays)
        if (!a) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    for (int32_t k = 0; k < T; ++k) {
        if (n[k] < 0) return fail(MICA_ERR_COUNT, "n[%d] = %lld is negative", k, (long long)n[k]);
        if (n[k] > ((int64_t)1 << 40)) return fail(MICA_ERR_COUNT, "n[%d] = %lld is too large", k, (long long)n[k]);
        if (n[k] == 0) continue;
        int j = 0;
        for (auto a : arrays) {
            if (!a[k]) return fail(MICA_ERR_NULL, "pointer %d of tensor %d is NULL (n = %lld)", j, k, (long long)n[k]);
            ++j;
        }
        *total += n[k];
    }
    return MICA_OK;
}

static mica_status current_device(int* dev) {
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(MICA_ERR_DEVICE, "no usable CUDA device (%s)", cudaGetErrorName(e));
    }
    return MICA_OK;
}

static bool finite_nonneg(double x) { return std::isfinite(x) && x >= 0.0; }

}  // namespace mica

using namespace mica;

// ----------------------------------------------------------------------------------------------------------------------
// entry points
// ----------------------------------------------------------------------------------------------------------------------

extern "C" mica_status mica_scale_tensors(void* const* t, const int64_t* n, int32_t T, mica_dtype dt, float factor,
                                          const float* d_factor, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (dt != MICA_F32 && dt != MICA_F16) return fail(MICA_ERR_DTYPE, "ScaleTensors takes float32 or float16 tensors");
    if (!d_factor && !std::isfinite(factor)) return fail(MICA_ERR_HYPER, "factor %g is not finite", (double)factor);
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!t || !n)) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    mica_status s;
    int dev = 0;
    ListDesc L{kScale, T, n, reinterpret_cast<float* const*>(t), nullptr, nullptr, nullptr, (Dtype)dt, kF32};
    Plan* p = nullptr;
    if (T > 0 && current_device(&dev) == MICA_OK) p = cached_plan(L, dev);
    if (!p) {
        int64_t total = 0;
        if ((s = check_list(T, n, {t}, &total)) != MICA_OK) return s;
        if (total == 0) return ok();
        if ((s = current_device(&dev)) != MICA_OK) return s;
        if ((s = get_plan(L, dev, &p, stream)) != MICA_OK) return s;
    }
    if ((s = check_scalars(p, dev, d_factor, nullptr, "one of the tensors")) != MICA_OK) return s;
    return after_launch(launch_scale(p->recs, p->items, p->num_items, p->item_octs, (Dtype)dt, factor, d_factor,
                                     stream),
                        stream, "ScaleTensors launch");
}

extern "C" mica_status mica_clip_grad_norms(const void* const* g, const int64_t* n, int32_t T, mica_dtype gdt,
                                            float max_norm, float inv_scale, float* d_norm, float* d_factor,
                                            void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (gdt != MICA_F32 && gdt != MICA_F16) return fail(MICA_ERR_DTYPE, "gradients must be float32 or float16");
    if (!d_factor) return fail(MICA_ERR_NULL, "d_factor is NULL");
    if (std::isnan(max_norm) || !(max_norm > 0.0f))
        return fail(MICA_ERR_HYPER, "max_norm %g is not > 0", (double)max_norm);
    if (!std::isfinite(inv_scale) || !(inv_scale > 0.0f))
        return fail(MICA_ERR_HYPER, "inv_scale %g is not finite and > 0", (double)inv_scale);
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!g || !n)) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    mica_status s;
    int dev = 0;
    ListDesc L{kNorm, T, n, nullptr, const_cast<void* const*>(reinterpret_cast<const void* const*>(g)), nullptr,
               nullptr, (Dtype)gdt, kF32};
    Plan* p = nullptr;
    if (T > 0 && current_device(&dev) == MICA_OK) p = cached_plan(L, dev);
    if (!p) {
        int64_t total = 0;
        if ((s = check_list(T, n, {g}, &total)) != MICA_OK) return s;
        if ((s = current_device(&dev)) != MICA_OK) return s;
        // An empty list still gets its norm (0) and factor written: its table holds no tensors.
        if (total == 0) L.T = 0;
        if ((s = get_plan(L, dev, &p, stream)) != MICA_OK) return s;
    }
    if ((s = check_scalars(p, dev, d_factor, d_norm, "a gradient")) != MICA_OK) return s;
    const bool keep_l2 = p->total * (int64_t)elem_bytes((Dtype)gdt) <= kKeepL2MaxGradBytes;
    return after_launch(launch_norm(p->chunks, (Dtype)gdt, inv_scale, p->partials, p->ticket, max_norm, d_norm,
                                    d_factor, nullptr, keep_l2, stream),
                        stream, "ClipGradNorms launch");
}

// The add g += a with the norm fused into it (both entry points below): the list's checks and cached table, then one
// launch writing d_norm / d_factor (the norm's call) or d_sumsq (one rank's square sum), each when not null.
static mica_status accumulate_call(void* const* g, const void* const* a, const int64_t* n, int32_t T, mica_dtype gdt,
                                   float max_norm, float inv_scale, float* d_norm, float* d_factor, double* d_sumsq,
                                   void* stream) {
    if (gdt != MICA_F32 && gdt != MICA_F16) return fail(MICA_ERR_DTYPE, "gradients must be float32 or float16");
    if (!std::isfinite(inv_scale) || !(inv_scale > 0.0f))
        return fail(MICA_ERR_HYPER, "inv_scale %g is not finite and > 0", (double)inv_scale);
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!g || !a || !n)) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    mica_status s;
    int dev = 0;
    ListDesc L{kAccNorm, T, n, nullptr, g, const_cast<void* const*>(reinterpret_cast<const void* const*>(a)),
               nullptr, (Dtype)gdt, kF32};
    Plan* p = nullptr;
    if (T > 0 && current_device(&dev) == MICA_OK) p = cached_plan(L, dev);
    if (!p) {
        int64_t total = 0;
        if ((s = check_list(T, n, {reinterpret_cast<const void* const*>(g), a}, &total)) != MICA_OK) return s;
        if ((s = current_device(&dev)) != MICA_OK) return s;
        if (total == 0) L.T = 0;  // an empty list still gets its outputs written
        if ((s = get_plan(L, dev, &p, stream)) != MICA_OK) return s;
    }
    if (d_sumsq) {
        if ((s = check_device_span(d_sumsq, 8, 8, dev, "d_sumsq", 0)) != MICA_OK) return s;
        if (overlaps_any(p->spans, d_sumsq, 8)) return fail(MICA_ERR_OVERLAP, "d_sumsq lies inside a gradient or an addend");
    } else if ((s = check_scalars(p, dev, d_factor, d_norm, "a gradient or an addend")) != MICA_OK) {
        return s;
    }
    const bool keep_l2 = p->total * (int64_t)elem_bytes((Dtype)gdt) <= kKeepL2MaxGradBytes;
    return after_launch(launch_accumulate_norm(p->chunks, (Dtype)gdt, inv_scale, p->partials, p->ticket, max_norm,
                                               d_norm, d_factor, d_sumsq, keep_l2, stream),
                        stream, d_sumsq ? "accumulating square-sum launch" : "AccumulateClipGradNorms launch");
}

extern "C" mica_status mica_accumulate_clip_grad_norms(void* const* g, const void* const* a, const int64_t* n,
                                                       int32_t T, mica_dtype gdt, float max_norm, float inv_scale,
                                                       float* d_norm, float* d_factor, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (!d_factor) return fail(MICA_ERR_NULL, "d_factor is NULL");
    if (std::isnan(max_norm) || !(max_norm > 0.0f))
        return fail(MICA_ERR_HYPER, "max_norm %g is not > 0", (double)max_norm);
    return accumulate_call(g, a, n, T, gdt, max_norm, inv_scale, d_norm, d_factor, nullptr, stream);
}

extern "C" mica_status mica_accumulate_grad_sumsq(void* const* g, const void* const* a, const int64_t* n, int32_t T,
                                                  mica_dtype gdt, float inv_scale, double* d_sumsq, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (!d_sumsq) return fail(MICA_ERR_NULL, "d_sumsq is NULL");
    return accumulate_call(g, a, n, T, gdt, 1.0f, inv_scale, nullptr, nullptr, d_sumsq, stream);
}

extern "C" mica_status mica_grad_sumsq(const void* const* g, const int64_t* n, int32_t T, mica_dtype gdt,
                                       float inv_scale, double* d_sumsq, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (gdt != MICA_F32 && gdt != MICA_F16) return fail(MICA_ERR_DTYPE, "gradients must be float32 or float16");
    if (!d_sumsq) return fail(MICA_ERR_NULL, "d_sumsq is NULL");
    if (!std::isfinite(inv_scale) || !(inv_scale > 0.0f))
        return fail(MICA_ERR_HYPER, "inv_scale %g is not finite and > 0", (double)inv_scale);
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!g || !n)) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    mica_status s;
    int dev = 0;
    ListDesc L{kNorm, T, n, nullptr, const_cast<void* const*>(reinterpret_cast<const void* const*>(g)), nullptr,
               nullptr, (Dtype)gdt, kF32};
    Plan* p = nullptr;
    if (T > 0 && current_device(&dev) == MICA_OK) p = cached_plan(L, dev);
    if (!p) {
        int64_t total = 0;
        if ((s = check_list(T, n, {g}, &total)) != MICA_OK) return s;
        if ((s = current_device(&dev)) != MICA_OK) return s;
        if (total == 0) L.T = 0;  // an empty list still gets its sum (0) written
        if ((s = get_plan(L, dev, &p, stream)) != MICA_OK) return s;
    }
    if ((s = check_device_span(d_sumsq, 8, 8, dev, "d_sumsq", 0)) != MICA_OK) return s;
    if (overlaps_any(p->spans, d_sumsq, 8)) return fail(MICA_ERR_OVERLAP, "d_sumsq lies inside a gradient");
    const bool keep_l2 = p->total * (int64_t)elem_bytes((Dtype)gdt) <= kKeepL2MaxGradBytes;
    return after_launch(launch_norm(p->chunks, (Dtype)gdt, inv_scale, p->partials, p->ticket, 1.0f, nullptr, nullptr,
                                    d_sumsq, keep_l2, stream),
                        stream, "square-sum launch");
}

extern "C" mica_status mica_clip_factor_from_sumsq(const double* d_parts, int32_t count, float max_norm,
                                                   float inv_scale, float* d_norm, float* d_factor, void* stream) {
    if (!d_parts || !d_factor) return fail(MICA_ERR_NULL, "d_parts or d_factor is NULL");
    if (count < 1 || count > (1 << 16)) return fail(MICA_ERR_COUNT, "count = %d is outside [1, 65536]", count);
    if (std::isnan(max_norm) || !(max_norm > 0.0f))
        return fail(MICA_ERR_HYPER, "max_norm %g is not > 0", (double)max_norm);
    if (!std::isfinite(inv_scale) || !(inv_scale > 0.0f))
        return fail(MICA_ERR_HYPER, "inv_scale %g is not finite and > 0", (double)inv_scale);
    int dev = 0;
    mica_status s = current_device(&dev);
    if (s != MICA_OK) return s;
    if ((s = check_device_span(d_parts, (size_t)count * 8, 8, dev, "d_parts", 0)) != MICA_OK) return s;
    if ((s = check_device_span(d_factor, 4, 4, dev, "d_factor", 0)) != MICA_OK) return s;
    if (d_norm && (s = check_device_span(d_norm, 4, 4, dev, "d_norm", 0)) != MICA_OK) return s;
    return after_launch(launch_factor_from_sumsq(d_parts, count, max_norm, inv_scale, d_norm, d_factor, stream), stream,
                        "factor launch");
}

namespace mica {

static mica_status check_adam_hp(const mica_adamw_hp* hp, int32_t j) {
    if (!finite_nonneg(hp->lr)) return fail(MICA_ERR_HYPER, "hp[%d].lr %g is not finite and >= 0", j, hp->lr);
    if (!finite_nonneg(hp->eps)) return fail(MICA_ERR_HYPER, "hp[%d].eps %g is not finite and >= 0", j, hp->eps);
    if (!finite_nonneg(hp->weight_decay))
        return fail(MICA_ERR_HYPER, "hp[%d].weight_decay %g is not finite and >= 0", j, hp->weight_decay);
    if (hp->step < 1) return fail(MICA_ERR_HYPER, "hp[%d].step %lld is not >= 1", j, (long long)hp->step);
    if (hp->flags & ~(MICA_STEP_SKIP_NONFINITE | MICA_STEP_COUPLED_L2))
        return fail(MICA_ERR_HYPER, "hp[%d].flags has unknown bits (0x%x)", j, hp->flags);
    if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0))
        return fail(MICA_ERR_BETA, "hp[%d].beta1 %g is outside [0, 1)", j, hp->beta1);
    if (!(hp->beta2 >= 0.0 && hp->beta2 < 1.0))
        return fail(MICA_ERR_BETA, "hp[%d].beta2 %g is outside [0, 1)", j, hp->beta2);
    return MICA_OK;
}

// What an AdamW launch needs, once its arguments have been checked: the list's table (null when the list holds no
// element), the current device and the step's scalars.
struct AdamCall {
    Plan* p = nullptr;
    int dev = 0;
    StepScalars sc{};
    GroupScalars gs{};
    bool coupled = false;
};

// The checks and the scalars of AdamWSteps with num_groups >= 1 parameter groups (group == nullptr: one group, every
// tensor in it); the list's table is found or built.
static mica_status prepare_adamw(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n,
                                 int32_t T, mica_dtype gdt, mica_dtype mdt, const int32_t* group,
                                 const mica_adamw_hp* hp, int32_t num_groups, const float* d_factor,
                                 const float* d_norm, void* stream, AdamCall* out) {
    if (!hp) return fail(MICA_ERR_NULL, "hp is NULL");
    if (gdt != MICA_F32 && gdt != MICA_F16) return fail(MICA_ERR_DTYPE, "gradients must be float32 or float16");
    if (mdt != MICA_F32 && mdt != MICA_BF16X2 && mdt != MICA_BF16X2_M)
        return fail(MICA_ERR_DTYPE, "moments must be float32, packed BF16, or packed m with float32 v");
    mica_status s;
    for (int32_t j = 0; j < num_groups; ++j) {
        if ((s = check_adam_hp(&hp[j], j)) != MICA_OK) return s;
        const mica_adamw_hp& a = hp[j];
        const mica_adamw_hp& z = hp[0];
        if (a.beta1 != z.beta1 || a.beta2 != z.beta2 || a.eps != z.eps || a.step != z.step ||
            (a.zero_grad != 0) != (z.zero_grad != 0) || a.flags != z.flags)
            return fail(MICA_ERR_HYPER, "hp[%d] differs from hp[0] in beta1, beta2, eps, step, zero_grad or flags "
                        "(only lr and weight_decay may differ between groups)", j);
    }
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!w || !g || !m || !v || !n)) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    int dev = 0;
    ListDesc L{kAdamW, T, n, w, g, m, v, (Dtype)gdt, (Dtype)mdt, group};
    Plan* p = nullptr;
    if (T > 0 && current_device(&dev) == MICA_OK) p = cached_plan(L, dev);
    if (!p) {
        int64_t total = 0;
        if ((s = check_list(T, n, {reinterpret_cast<const void* const*>(w), g, m, v}, &total)) != MICA_OK) return s;
        if (group)
            for (int32_t k = 0; k < T; ++k)
                if (group[k] < 0 || group[k] >= num_groups)
                    return fail(MICA_ERR_COUNT, "group[%d] = %d is outside [0, %d)", k, group[k], num_groups);
        if (total == 0) {
            out->p = nullptr;
            return ok();
        }
        if ((s = current_device(&dev)) != MICA_OK) return s;
        if ((s = get_plan(L, dev, &p, stream)) != MICA_OK) return s;
    }
    if (p->total == 0) {
        out->p = nullptr;
        return ok();
    }
    if (group && p->max_group >= num_groups)  // a list seen before with more groups
        return fail(MICA_ERR_COUNT, "group index %d is outside [0, %d)", p->max_group, num_groups);
    if ((s = check_scalars(p, dev, d_factor, d_norm, "one of the step's buffers")) != MICA_OK) return s;

    // the step's scalars: PyTorch's, each in double and rounded once to float32
    const double t = (double)hp->step;
    const double q1 = 1.0 - std::pow(hp->beta1, t);
    StepScalars& sc = out->sc;
    sc = StepScalars{};
    sc.c1 = (float)(1.0 - hp->beta1);
    sc.b2 = (float)hp->beta2;
    sc.c2 = (float)(1.0 - hp->beta2);
    sc.neg_step = -(float)(hp->lr / q1);
    sc.bc2 = (float)std::sqrt(1.0 - std::pow(hp->beta2, t));
    sc.dec = (float)(1.0 - hp->lr * hp->weight_decay);
    sc.eps = (float)hp->eps;
    sc.wd = (float)hp->weight_decay;
    sc.zero_grad = hp->zero_grad ? 1 : 0;
    sc.skip_nonfinite = (hp->flags & MICA_STEP_SKIP_NONFINITE) ? 1 : 0;
    out->coupled = (hp->flags & MICA_STEP_COUPLED_L2) != 0;
    out->gs = GroupScalars{};
    for (int32_t j = 0; j < num_groups; ++j) {
        out->gs.neg_step[j] = -(float)(hp[j].lr / q1);
        out->gs.dec[j] = (float)(1.0 - hp[j].lr * hp[j].weight_decay);
        out->gs.wd[j] = (float)hp[j].weight_decay;
    }
    out->p = p;
    out->dev = dev;
    return MICA_OK;
}

// AdamWSteps with num_groups >= 1 parameter groups (group == nullptr: one group, every tensor in it).
static mica_status adamw_steps(float* const* w, void* const* g, void* const* m, void* const* v, const int64_t* n,
                               int32_t T, mica_dtype gdt, mica_dtype mdt, const int32_t* group,
                               const mica_adamw_hp* hp, int32_t num_groups, const float* d_factor, void* stream) {
    AdamCall a;
    const mica_status s = prepare_adamw(w, g, m, v, n, T, gdt, mdt, group, hp, num_groups, d_factor, nullptr, stream,
                                        &a);
    if (s != MICA_OK || !a.p) return s;
    return after_launch(launch_adamw(update_launch(a.p, true), (Dtype)gdt, (Dtype)mdt, a.coupled, a.sc,
                                     group ? &a.gs : nullptr, d_factor, stream),
                        stream, "AdamWSteps launch");
}

// Whether mica_clip_adamw_step runs the norm and the update as one cooperative launch: only when MICA_FUSED=1 (read
// at each call). Measured on GB300, the two launches chained by programmatic dependent launch are faster for every
// list tried (the loss-scaled list of 10,012 tensors: 0.196 against 0.202 ms a step; the tiny list: 0.017 against
// 0.021 ms), because a cooperative launch cannot overlap the steps before and after it, and its norm phase runs at
// the update's 3 CTAs per SM; the two launches get the L2 re-read too, from the norm's evict-last policy on
// gradients that fit in L2.
static bool use_fused() {
    const char* e = std::getenv("MICA_FUSED");
    return e && std::strcmp(e, "1") == 0;
}

}  // namespace mica

extern "C" mica_status mica_adamw_steps(float* const* w, void* const* g, void* const* m, void* const* v,
                                        const int64_t* n, int32_t T, mica_dtype gdt, mica_dtype mdt,
                                        const mica_adamw_hp* hp, const float* d_factor, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    return adamw_steps(w, g, m, v, n, T, gdt, mdt, nullptr, hp, 1, d_factor, stream);
}

extern "C" mica_status mica_adamw_steps_grouped(float* const* w, void* const* g, void* const* m, void* const* v,
                                                const int64_t* n, int32_t T, mica_dtype gdt, mica_dtype mdt,
                                                const int32_t* group, const mica_adamw_hp* hp, int32_t num_groups,
                                                const float* d_factor, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (num_groups < 1 || num_groups > MICA_MAX_GROUPS)
        return fail(MICA_ERR_COUNT, "num_groups = %d is outside [1, %d]", num_groups, MICA_MAX_GROUPS);
    if (T > 0 && !group) return fail(MICA_ERR_NULL, "group is NULL");
    return adamw_steps(w, g, m, v, n, T, gdt, mdt, T > 0 ? group : nullptr, hp, num_groups, d_factor, stream);
}

extern "C" mica_status mica_clip_adamw_step(float* const* w, void* const* g, void* const* m, void* const* v,
                                            const int64_t* n, int32_t T, mica_dtype gdt, mica_dtype mdt,
                                            const mica_adamw_hp* hp, float max_norm, float inv_scale, float* d_norm,
                                            float* d_factor, void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    // the norm's own checks (those of mica_clip_grad_norms), then the update's (those of mica_adamw_steps)
    if (gdt != MICA_F32 && gdt != MICA_F16) return fail(MICA_ERR_DTYPE, "gradients must be float32 or float16");
    if (!d_factor) return fail(MICA_ERR_NULL, "d_factor is NULL");
    if (std::isnan(max_norm) || !(max_norm > 0.0f))
        return fail(MICA_ERR_HYPER, "max_norm %g is not > 0", (double)max_norm);
    if (!std::isfinite(inv_scale) || !(inv_scale > 0.0f))
        return fail(MICA_ERR_HYPER, "inv_scale %g is not finite and > 0", (double)inv_scale);
    AdamCall a;
    mica_status s = prepare_adamw(w, g, m, v, n, T, gdt, mdt, nullptr, hp, 1, d_factor, d_norm, stream, &a);
    if (s != MICA_OK) return s;
    // the two launches of mica_clip_grad_norms and mica_adamw_steps (an empty list only gets its norm, 0, and its
    // factor, inv_scale)
    auto two_launches = [&]() -> mica_status {
        mica_status r = mica_clip_grad_norms(const_cast<const void* const*>(g), n, T, gdt, max_norm, inv_scale, d_norm,
                                             d_factor, stream);
        if (r != MICA_OK || !a.p) return r;
        return after_launch(launch_adamw(update_launch(a.p, true), (Dtype)gdt, (Dtype)mdt, a.coupled, a.sc, nullptr,
                                         d_factor, stream),
                            stream, "AdamWSteps launch");
    };
    if (!a.p || !use_fused()) return two_launches();
    if ((s = ensure_fused_table(a.p, stream)) != MICA_OK) return s;
    const int e = launch_clip_adamw(a.p->fchunks, a.p->fpartials, a.p->fbar, update_launch(a.p, true, true),
                                    (Dtype)gdt, (Dtype)mdt, a.coupled, a.sc, max_norm, inv_scale, d_norm, d_factor,
                                    stream);
    if (e == (int)cudaErrorCooperativeLaunchTooLarge) {  // not one wave on this GPU: nothing queued, two launches
        cudaGetLastError();
        return two_launches();
    }
    return after_launch(e, stream, "fused ClipGradNorms + AdamWSteps launch");
}

extern "C" mica_status mica_sgd_steps(float* const* w, void* const* g, float* const* buf, const int64_t* n,
                                      int32_t T, mica_dtype gdt, const mica_sgd_hp* hp, const float* d_factor,
                                      void* stream) {
    CallScope scope;  // the tables this call looks up stay pinned until it returns
    if (!hp) return fail(MICA_ERR_NULL, "hp is NULL");
    if (gdt != MICA_F32 && gdt != MICA_F16) return fail(MICA_ERR_DTYPE, "gradients must be float32 or float16");
    if (!finite_nonneg(hp->lr)) return fail(MICA_ERR_HYPER, "lr %g is not finite and >= 0", hp->lr);
    if (!finite_nonneg(hp->momentum)) return fail(MICA_ERR_HYPER, "momentum %g is not finite and >= 0", hp->momentum);
    if (!buf && hp->momentum != 0.0) return fail(MICA_ERR_NULL, "momentum %g > 0 needs the buffer array", hp->momentum);
    if (hp->flags & ~MICA_STEP_SKIP_NONFINITE)
        return fail(MICA_ERR_HYPER, "hp->flags has bits SGD does not take (0x%x)", hp->flags);
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!w || !g || !n)) return fail(MICA_ERR_NULL, "a pointer array is NULL");
    mica_status s;
    int dev = 0;
    const Kind kind = buf ? kMomentum : kSGD;
    ListDesc L{kind, T, n, w, g, reinterpret_cast<void* const*>(buf), nullptr, (Dtype)gdt, kF32};
    Plan* p = nullptr;
    if (T > 0 && current_device(&dev) == MICA_OK) p = cached_plan(L, dev);
    if (!p) {
        int64_t total = 0;
        if (buf)
            s = check_list(T, n, {reinterpret_cast<const void* const*>(w), g,
                                  reinterpret_cast<const void* const*>(buf)}, &total);
        else
            s = check_list(T, n, {reinterpret_cast<const void* const*>(w), g}, &total);
        if (s != MICA_OK) return s;
        if (total == 0) return ok();
        if ((s = current_device(&dev)) != MICA_OK) return s;
        if ((s = get_plan(L, dev, &p, stream)) != MICA_OK) return s;
    }
    if (p->total == 0) return ok();
    if ((s = check_scalars(p, dev, d_factor, nullptr, "one of the step's buffers")) != MICA_OK) return s;
    SgdScalars sc{};
    sc.neg_lr = -(float)hp->lr;
    sc.mu = (float)hp->momentum;
    sc.zero_grad = hp->zero_grad ? 1 : 0;
    // plain SGD's short update keeps the next norm waiting less when each item is its own CTA (measured)
    return after_launch(launch_sgd(update_launch(p, buf != nullptr), (Dtype)gdt, buf != nullptr,
                                   (hp->flags & MICA_STEP_SKIP_NONFINITE) != 0, sc, d_factor, stream),
                        stream, "SGDSteps launch");
}

extern "C" mica_status mica_selftest_wait_timeout(uint32_t polls, void* stream) {
    if (polls < 1 || polls > (1u << 20)) return fail(MICA_ERR_HYPER, "polls = %u is outside [1, 2^20]", polls);
    int dev = 0;
    mica_status s = current_device(&dev);
    if (s != MICA_OK) return s;
    return after_launch(launch_wait_selftest(polls, stream), stream, "wait self-test launch");
}

extern "C" mica_status mica_selftest_grid_wait_timeout(uint32_t polls, void* stream) {
    if (polls < 1 || polls > (1u << 20)) return fail(MICA_ERR_HYPER, "polls = %u is outside [1, 2^20]", polls);
    int dev = 0;
    mica_status s = current_device(&dev);
    if (s != MICA_OK) return s;
    return after_launch(launch_grid_wait_selftest(polls, stream), stream, "grid-wait self-test launch");
}

extern "C" mica_status mica_sync(void* stream) {
    const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "mica_sync");
    const mica_status s = check_device_status("mica_sync");
    if (s != MICA_OK) return s;
    return ok();
}

extern "C" mica_status mica_release_cache(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    cudaError_t e = cudaSuccess;
    if (g_plan_count) e = cudaDeviceSynchronize();
    evict_unpinned();
    noalloc_forget_addresses();
    if (e != cudaSuccess) return cuda_fail(e, "mica_release_cache");
    return ok();
}

extern "C" const char* mica_status_string(mica_status s) {
    switch (s) {
        case MICA_OK: return "MICA_OK";
        case MICA_ERR_NULL: return "MICA_ERR_NULL";
        case MICA_ERR_COUNT: return "MICA_ERR_COUNT";
        case MICA_ERR_DTYPE: return "MICA_ERR_DTYPE";
        case MICA_ERR_HYPER: return "MICA_ERR_HYPER";
        case MICA_ERR_BETA: return "MICA_ERR_BETA";
        case MICA_ERR_OVERLAP: return "MICA_ERR_OVERLAP";
        case MICA_ERR_DEVICE: return "MICA_ERR_DEVICE";
        case MICA_ERR_ADDRESS: return "MICA_ERR_ADDRESS";
        case MICA_ERR_CUDA: return "MICA_ERR_CUDA";
        case MICA_ERR_NOMEM: return "MICA_ERR_NOMEM";
        case MICA_ERR_CAPTURE: return "MICA_ERR_CAPTURE";
    }
    return "MICA_ERR_UNKNOWN";
}

extern "C" const char* mica_last_error_detail(void) { return t_detail.c_str(); }

extern "C" uint64_t mica_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" mica_status mica_work_items(const int64_t* n, const int32_t* vec, int32_t T, int32_t item_octs,
                                       int32_t sms, int64_t* items, int32_t max_items, int32_t* pack,
                                       int32_t max_pack, int32_t* num_items, int32_t* pack_len,
                                       int32_t* used_item_octs) {
    if (!num_items || !pack_len) return fail(MICA_ERR_NULL, "num_items and pack_len must not be NULL");
    if (T < 0 || T > MICA_MAX_TENSORS) return fail(MICA_ERR_COUNT, "T = %d is outside [0, %d]", T, MICA_MAX_TENSORS);
    if (T > 0 && (!n || !vec)) return fail(MICA_ERR_NULL, "n and vec must not be NULL");
    if (max_items < 0 || max_pack < 0) return fail(MICA_ERR_COUNT, "a capacity is negative");
    if ((max_items > 0 && !items) || (max_pack > 0 && !pack))
        return fail(MICA_ERR_NULL, "an output array is NULL but its capacity is not 0");
    if (sms < 1) return fail(MICA_ERR_COUNT, "sms = %d is not >= 1", sms);
    if (item_octs != 0 && (item_octs < 16 || item_octs > (1 << 20) || (item_octs & (item_octs - 1)) != 0))
        return fail(MICA_ERR_COUNT, "item_octs = %d is not 0 or a power of two in [16, 2^20]", item_octs);
    std::vector<TensorRec> recs((size_t)T);
    int64_t total_octs = 0;
    for (int32_t k = 0; k < T; ++k) {
        if (n[k] < 0 || n[k] > ((int64_t)1 << 40))
            return fail(MICA_ERR_COUNT, "n[%d] = %lld is outside [0, 2^40]", k, (long long)n[k]);
        recs[(size_t)k] = TensorRec{nullptr, nullptr, nullptr, nullptr, n[k], vec[k] ? 1 : 0, 0};
        total_octs += (n[k] + kOct - 1) / kOct;
    }
    const int32_t io = item_octs ? item_octs : choose_item_octs(total_octs, sms, base_item_octs(kAdamW, kF32));
    std::vector<int32_t> pre;
    std::vector<WorkItem> list = build_items(n, recs.data(), T, io, &pre);
    order_items(list);
    if (list.size() > (size_t)INT32_MAX || pre.size() > (size_t)INT32_MAX)
        return fail(MICA_ERR_COUNT, "too many work items (%zu)", list.size());
    *num_items = (int32_t)list.size();
    *pack_len = (int32_t)pre.size();
    if (used_item_octs) *used_item_octs = io;
    for (size_t i = 0; i < list.size() && i < (size_t)max_items; ++i) {
        items[3 * i] = list[i].t;
        items[3 * i + 1] = list[i].count;
        items[3 * i + 2] = list[i].o0;
    }
    for (size_t i = 0; i < pre.size() && i < (size_t)max_pack; ++i) pack[i] = pre[i];
    return ok();
}

extern "C" int32_t mica_abi_version(void) { return 5; }
