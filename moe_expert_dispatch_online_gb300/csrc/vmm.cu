// Weight store for the "VM group GEMM" contract, with CUDA virtual memory
// management (cuMemCreate / cuMemMap) on one GPU.
//
// MoonEP pages (ai-maestro.online), "The memory contract": each expert
// projection is one contiguous [E+B, H, H'] tensor per rank; rows [0, E) are
// every rank's home experts, each chunk physically the home rank's parameter
// memory mapped everywhere; rows [E, E+B) are the rank's prefetch slots, drawn
// from a process-global pool shared by all layers, so the extra cost is B
// experts per projection in total, not per layer.
//
// Here the R virtual ranks share one GPU, so "mapped everywhere" becomes
// aliasing inside one address space:
//   * per layer l, one physical block holds the home rows [E, H, H'];
//   * the slot pool [R, B, H, H'] (one physical block per rank), shared by layers;
//   * per layer, R views [E+B, H, H'] are placed back to back: view u maps the
//     layer's home block at rows [0, E) and rank u's part of the pool at rows
//     [E, E+B). No byte is copied; a write through any alias is seen by all.
// The driver maps a physical block only whole, so the home rows of a layer
// (E*H*H'*2 bytes) and one rank's slots (B*H*H'*2 bytes) must each be a
// multiple of the mapping granularity (2 MiB on this GPU); otherwise
// bep_weights_create returns BEP_ERR_SIZE.

#include <cuda.h>
#include <stdio.h>
#include <stdlib.h>

#include <vector>

#include "bep_internal.cuh"

namespace {

struct Drv {
    decltype(&cuMemCreate) create = nullptr;
    decltype(&cuMemRelease) release = nullptr;
    decltype(&cuMemAddressReserve) reserve = nullptr;
    decltype(&cuMemAddressFree) addr_free = nullptr;
    decltype(&cuMemMap) map = nullptr;
    decltype(&cuMemUnmap) unmap = nullptr;
    decltype(&cuMemSetAccess) set_access = nullptr;
    decltype(&cuMemGetAllocationGranularity) granularity = nullptr;
    bool ok = false;
};

template <typename F>
bool entry(const char* name, F* fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Drv& drv() {
    static Drv d = [] {
        Drv x;
        x.ok = entry("cuMemCreate", &x.create) && entry("cuMemRelease", &x.release) &&
               entry("cuMemAddressReserve", &x.reserve) && entry("cuMemAddressFree", &x.addr_free) &&
               entry("cuMemMap", &x.map) && entry("cuMemUnmap", &x.unmap) &&
               entry("cuMemSetAccess", &x.set_access) &&
               entry("cuMemGetAllocationGranularity", &x.granularity);
        return x;
    }();
    return d;
}

// With BEP_DEBUG set in the environment, a failing driver call is reported on
// stderr (the C ABI itself only returns BEP_ERR_CUDA).
bool check(CUresult r, const char* what) {
    if (r == CUDA_SUCCESS) return true;
    if (getenv("BEP_DEBUG")) fprintf(stderr, "bep_weights_create: %s failed (CUresult %d)\n", what, (int)r);
    return false;
}

struct Range {
    CUdeviceptr va;
    size_t size;
};

}  // namespace

struct bep_weights {
    bep::Dims d;
    int device;
    int layers;
    size_t row_bytes;
    std::vector<CUmemGenericAllocationHandle> handles;   // layers home blocks, then R pool blocks
    std::vector<Range> reserved;                         // every reserved VA range
    std::vector<Range> mapped;                           // every mapping, for unmapping
    std::vector<uint16_t*> home;                         // per layer [E, H, H']
    uint16_t* slots = nullptr;                           // [R, B, H, H']
    std::vector<uint16_t*> views;                        // per layer [R, E+B, H, H']
};

namespace {

void teardown(bep_weights* w) {
    const Drv& D = drv();
    for (const Range& m : w->mapped) D.unmap(m.va, m.size);
    for (const Range& r : w->reserved) D.addr_free(r.va, r.size);
    for (CUmemGenericAllocationHandle h : w->handles) D.release(h);
    delete w;
}

bool reserve_and_access(bep_weights* w, size_t size, CUdeviceptr* va) {
    const Drv& D = drv();
    if (!check(D.reserve(va, size, 0, 0, 0), "cuMemAddressReserve")) return false;
    w->reserved.push_back({*va, size});
    return true;
}

bool map_at(bep_weights* w, CUdeviceptr va, size_t size, size_t offset,
            CUmemGenericAllocationHandle h) {
    if (!check(drv().map(va, size, offset, h, 0), "cuMemMap")) return false;
    w->mapped.push_back({va, size});
    return true;
}

bool set_rw(bep_weights* w, CUdeviceptr va, size_t size) {
    CUmemAccessDesc a = {};
    a.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    a.location.id = w->device;
    a.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    return check(drv().set_access(va, size, &a, 1), "cuMemSetAccess");
}

}  // namespace

extern "C" {

int bep_weights_create(const bep_config* cfg, int32_t layers, bep_weights** out) {
    if (!cfg || !out || layers < 1) return BEP_ERR_ARG;
    *out = nullptr;
    bep::Dims d;
    const int rc = bep::make_dims(cfg, &d);
    if (rc) return rc;
    if (d.B < 1) return BEP_ERR_SIZE;
    const Drv& D = drv();
    if (!D.ok) {
        if (getenv("BEP_DEBUG")) fprintf(stderr, "bep_weights_create: driver entry points missing\n");
        return BEP_ERR_CUDA;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BEP_ERR_CUDA;
    // make sure the runtime has made the device's primary context current
    if (cudaFree(nullptr) != cudaSuccess) return BEP_ERR_CUDA;

    CUmemAllocationProp prop = {};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = dev;
    size_t gran = 0;
    if (!check(D.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM),
               "cuMemGetAllocationGranularity") || !gran)
        return BEP_ERR_CUDA;
    const size_t row = (size_t)d.H * d.Hp * sizeof(uint16_t);
    if ((row * d.E) % gran != 0 || (row * d.B) % gran != 0) return BEP_ERR_SIZE;

    bep_weights* w = new bep_weights;
    w->d = d;
    w->device = dev;
    w->layers = layers;
    w->row_bytes = row;
    const size_t home_bytes = row * d.E, pool_bytes = row * (size_t)d.R * d.B;
    const size_t view_bytes = row * (size_t)(d.E + d.B);
    auto fail = [&](int code) {
        teardown(w);
        return code;
    };
    // physical blocks: the layers' home rows, then the pool as one block per rank
    // (the driver maps a physical block only whole, from offset 0)
    const size_t rank_pool_bytes = row * (size_t)d.B;
    for (int l = 0; l < layers + d.R; ++l) {
        CUmemGenericAllocationHandle h;
        if (!check(D.create(&h, l < layers ? home_bytes : rank_pool_bytes, &prop, 0), "cuMemCreate"))
            return fail(BEP_ERR_CUDA);
        w->handles.push_back(h);
    }
    auto pool = [&](int u) { return w->handles[layers + u]; };
    // the pool, as [R, B, H, H']
    CUdeviceptr va;
    if (!reserve_and_access(w, pool_bytes, &va)) return fail(BEP_ERR_CUDA);
    for (int u = 0; u < d.R; ++u)
        if (!map_at(w, va + rank_pool_bytes * u, rank_pool_bytes, 0, pool(u)))
            return fail(BEP_ERR_CUDA);
    if (!set_rw(w, va, pool_bytes)) return fail(BEP_ERR_CUDA);
    w->slots = reinterpret_cast<uint16_t*>(va);
    for (int l = 0; l < layers; ++l) {
        const CUmemGenericAllocationHandle h = w->handles[l];
        // the layer's home rows, as [E, H, H']
        if (!reserve_and_access(w, home_bytes, &va) || !map_at(w, va, home_bytes, 0, h) ||
            !set_rw(w, va, home_bytes))
            return fail(BEP_ERR_CUDA);
        w->home.push_back(reinterpret_cast<uint16_t*>(va));
        // R views back to back: home rows (aliased) then rank u's slots
        if (!reserve_and_access(w, view_bytes * d.R, &va)) return fail(BEP_ERR_CUDA);
        for (int u = 0; u < d.R; ++u) {
            const CUdeviceptr base = va + view_bytes * u;
            if (!map_at(w, base, home_bytes, 0, h) ||
                !map_at(w, base + home_bytes, rank_pool_bytes, 0, pool(u)))
                return fail(BEP_ERR_CUDA);
        }
        if (!set_rw(w, va, view_bytes * d.R)) return fail(BEP_ERR_CUDA);
        w->views.push_back(reinterpret_cast<uint16_t*>(va));
    }
    *out = w;
    return BEP_OK;
}

int bep_weights_get(bep_weights* w, int32_t layer, uint16_t** home, uint16_t** slots,
                    uint16_t** views) {
    if (!w || layer < 0 || layer >= w->layers) return BEP_ERR_ARG;
    if (home) *home = w->home[layer];
    if (slots) *slots = w->slots;
    if (views) *views = w->views[layer];
    return BEP_OK;
}

void bep_weights_destroy(bep_weights* w) {
    if (!w) return;
    teardown(w);
}

}  // extern "C"
