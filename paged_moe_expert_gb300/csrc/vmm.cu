// A contiguous virtual view over scattered physical blocks (CUDA driver virtual memory
// management), the rival design to looking pages up inside the kernel: FluxMoE
// (awesome-system-papers, section "核心方法", PagedTensor) keeps a stable virtual address per
// weight tensor and maps physical blocks under it before the kernel runs.  Host code only.
#include <chrono>
#include <thread>
#include <vector>

#include "pmoe_internal.cuh"

struct pmoe_vmm {
    int device = 0;
    size_t block_bytes = 0;
    int64_t n_blocks = 0, n_virtual = 0;
    std::vector<CUmemGenericAllocationHandle> handles;
    CUdeviceptr blocks = 0, view = 0;
    int64_t blocks_mapped = 0;            // blocks mapped in the `blocks` range (0..n_blocks)
    std::vector<int64_t> block_of;        // [n_virtual]: block under each virtual page, or -1
};

namespace {

struct VmmApi {
    CUresult (*granularity)(size_t*, const CUmemAllocationProp*, CUmemAllocationGranularity_flags);
    CUresult (*create)(CUmemGenericAllocationHandle*, size_t, const CUmemAllocationProp*,
                       unsigned long long);
    CUresult (*release)(CUmemGenericAllocationHandle);
    CUresult (*reserve)(CUdeviceptr*, size_t, size_t, CUdeviceptr, unsigned long long);
    CUresult (*free_range)(CUdeviceptr, size_t);
    CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long);
    CUresult (*unmap)(CUdeviceptr, size_t);
    CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc*, size_t);
    bool ok = false;
};

template <typename F>
bool entry(const char* name, F& fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    fn = reinterpret_cast<F>(p);
    return true;
}

const VmmApi& api() {
    static VmmApi a = [] {
        VmmApi v{};
        v.ok = entry("cuMemGetAllocationGranularity", v.granularity) &&
               entry("cuMemCreate", v.create) && entry("cuMemRelease", v.release) &&
               entry("cuMemAddressReserve", v.reserve) && entry("cuMemAddressFree", v.free_range) &&
               entry("cuMemMap", v.map) && entry("cuMemUnmap", v.unmap) &&
               entry("cuMemSetAccess", v.set_access);
        return v;
    }();
    return a;
}

CUmemAllocationProp device_prop(int device) {
    CUmemAllocationProp p{};
    p.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    p.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    p.location.id = device;
    return p;
}

pmoe_status bad(pmoe_status s, const char* msg) { return pmoe::record_failure(s, msg); }

pmoe_status drv(CUresult r, const char* what) {
    return r == CUDA_SUCCESS ? PMOE_OK : pmoe::record_failure(PMOE_ERR_CUDA, what);
}

// Makes the runtime's context of `device` current for the driver calls that follow, and puts the
// caller's current device back when it goes out of scope.
struct DeviceScope {
    int prev = -1;
    pmoe_status status = PMOE_OK;
    explicit DeviceScope(int device) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (cudaSetDevice(device) != cudaSuccess || cudaFree(nullptr) != cudaSuccess)
            status = bad(PMOE_ERR_CUDA, "pmoe_vmm: cannot make the device current");
    }
    ~DeviceScope() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

pmoe_status map_one(pmoe_vmm* v, CUdeviceptr at, CUmemGenericAllocationHandle h) {
    const VmmApi& A = api();
    pmoe_status st = drv(A.map(at, v->block_bytes, 0, h, 0), "cuMemMap failed");
    if (st != PMOE_OK) return st;
    CUmemAccessDesc acc{};
    acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc.location.id = v->device;
    acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    st = drv(A.set_access(at, v->block_bytes, &acc, 1), "cuMemSetAccess failed");
    if (st != PMOE_OK) A.unmap(at, v->block_bytes);
    return st;
}

void teardown(pmoe_vmm* v) {
    const VmmApi& A = api();
    if (v->view) {
        for (int64_t i = 0; i < v->n_virtual; ++i)
            if (v->block_of[i] >= 0) A.unmap(v->view + (CUdeviceptr)(i * v->block_bytes), v->block_bytes);
        A.free_range(v->view, v->block_bytes * v->n_virtual);
    }
    if (v->blocks) {
        for (int64_t i = 0; i < v->blocks_mapped; ++i)
            A.unmap(v->blocks + (CUdeviceptr)(i * v->block_bytes), v->block_bytes);
        A.free_range(v->blocks, v->block_bytes * v->n_blocks);
    }
    for (CUmemGenericAllocationHandle h : v->handles) A.release(h);
    delete v;
}

}  // namespace

extern "C" pmoe_status pmoe_vmm_granularity(int32_t device, size_t* bytes) {
    if (!bytes) return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_granularity: bytes is NULL");
    *bytes = 0;
    if (!api().ok) return bad(PMOE_ERR_CUDA, "pmoe_vmm: driver VMM entry points not found");
    DeviceScope scope(device);
    if (scope.status != PMOE_OK) return scope.status;
    const CUmemAllocationProp p = device_prop(device);
    return drv(api().granularity(bytes, &p, CU_MEM_ALLOC_GRANULARITY_MINIMUM),
               "cuMemGetAllocationGranularity failed");
}

extern "C" pmoe_status pmoe_vmm_create(int32_t device, size_t block_bytes, int64_t n_blocks,
                                       int64_t n_virtual, pmoe_vmm_t* out) {
    if (!out) return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_create: out is NULL");
    *out = nullptr;
    if (block_bytes == 0 || n_blocks < 1 || n_virtual < 1)
        return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_create: block_bytes, n_blocks, n_virtual >= 1");
    DeviceScope scope(device);
    if (scope.status != PMOE_OK) return scope.status;
    size_t g = 0;
    pmoe_status st = pmoe_vmm_granularity(device, &g);
    if (st != PMOE_OK) return st;
    if (block_bytes % g != 0)
        return bad(PMOE_ERR_UNSUPPORTED, "pmoe_vmm_create: block_bytes is not a multiple of the "
                                         "VMM granularity");
    pmoe_vmm* v = new pmoe_vmm;
    v->device = device;
    v->block_bytes = block_bytes;
    v->n_blocks = n_blocks;
    v->n_virtual = n_virtual;
    v->block_of.assign(n_virtual, -1);
    const VmmApi& A = api();
    const CUmemAllocationProp p = device_prop(device);
    for (int64_t i = 0; i < n_blocks; ++i) {
        CUmemGenericAllocationHandle h;
        if ((st = drv(A.create(&h, block_bytes, &p, 0), "cuMemCreate failed")) != PMOE_OK) {
            teardown(v);
            return st;
        }
        v->handles.push_back(h);
    }
    if ((st = drv(A.reserve(&v->blocks, block_bytes * n_blocks, 0, 0, 0),
                  "cuMemAddressReserve failed")) != PMOE_OK ||
        (st = drv(A.reserve(&v->view, block_bytes * n_virtual, 0, 0, 0),
                  "cuMemAddressReserve failed")) != PMOE_OK) {
        teardown(v);
        return st;
    }
    for (int64_t i = 0; i < n_blocks; ++i) {
        if ((st = map_one(v, v->blocks + (CUdeviceptr)(i * block_bytes), v->handles[i])) != PMOE_OK) {
            teardown(v);
            return st;
        }
        v->blocks_mapped = i + 1;
    }
    *out = v;
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_vmm_destroy(pmoe_vmm_t v) {
    if (!v) return PMOE_OK;
    DeviceScope scope(v->device);
    if (scope.status != PMOE_OK) return scope.status;
    teardown(v);
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_vmm_pointers(pmoe_vmm_t v, void** blocks, void** view) {
    if (!v) return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_pointers: vmm is NULL");
    if (blocks) *blocks = reinterpret_cast<void*>(v->blocks);
    if (view) *view = reinterpret_cast<void*>(v->view);
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_vmm_map(pmoe_vmm_t v, int64_t n, const int64_t* virt,
                                    const int64_t* blocks) {
    if (!v || n < 0 || (n > 0 && (!virt || !blocks)))
        return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_map: vmm non-NULL, n >= 0, arrays non-NULL");
    std::vector<uint8_t> seen(v->n_virtual, 0);
    for (int64_t i = 0; i < n; ++i) {
        if (virt[i] < 0 || virt[i] >= v->n_virtual || blocks[i] < 0 || blocks[i] >= v->n_blocks)
            return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_map: page or block out of range");
        if (v->block_of[virt[i]] >= 0 || seen[virt[i]])
            return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_map: virtual page already mapped or listed twice");
        seen[virt[i]] = 1;
    }
    DeviceScope scope(v->device);
    if (scope.status != PMOE_OK) return scope.status;
    pmoe_status st = PMOE_OK;
    for (int64_t i = 0; i < n; ++i) {
        st = map_one(v, v->view + (CUdeviceptr)(virt[i] * v->block_bytes), v->handles[blocks[i]]);
        if (st != PMOE_OK) return st;   // the pages before i stay mapped (pmoe_vmm_lookup shows them)
        v->block_of[virt[i]] = blocks[i];
    }
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_vmm_unmap(pmoe_vmm_t v, int64_t n, const int64_t* virt,
                                      pmoe_event_t readers_done, int32_t timeout_ms) {
    if (!v || n < 0 || (n > 0 && !virt))
        return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_unmap: vmm non-NULL, n >= 0, virt non-NULL");
    for (int64_t i = 0; i < n; ++i)
        if (virt[i] < 0 || virt[i] >= v->n_virtual || v->block_of[virt[i]] < 0)
            return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_unmap: page out of range or not mapped");
    if (readers_done) {
        pmoe_status st = pmoe_wait_event(readers_done, timeout_ms);
        if (st != PMOE_OK) return st;
    }
    DeviceScope scope(v->device);
    if (scope.status != PMOE_OK) return scope.status;
    pmoe_status st = PMOE_OK;
    for (int64_t i = 0; i < n; ++i) {
        if (v->block_of[virt[i]] < 0) continue;   // listed twice
        st = drv(api().unmap(v->view + (CUdeviceptr)(virt[i] * v->block_bytes), v->block_bytes),
                 "cuMemUnmap failed");
        if (st != PMOE_OK) return st;
        v->block_of[virt[i]] = -1;
    }
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_vmm_lookup(pmoe_vmm_t v, int64_t* block_of) {
    if (!v || !block_of) return bad(PMOE_ERR_INVALID_ARG, "pmoe_vmm_lookup: NULL argument");
    for (int64_t i = 0; i < v->n_virtual; ++i) block_of[i] = v->block_of[i];
    return PMOE_OK;
}
