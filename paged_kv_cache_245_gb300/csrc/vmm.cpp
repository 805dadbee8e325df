// vmm.cpp -- contiguous per-request KV buffers whose physical memory is
// mapped on demand through the CUDA virtual memory management calls
// ("Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory": one
// large virtual range per layer holds every request's sub-tensor at offset
// reqId x S; physical pages are mapped into it as a request's context grows,
// and unmapped when the request ends).  Host code; the driver entry points
// are looked up at run time, so the library links no driver library.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <mutex>
#include <new>
#include <vector>

#include "pkv_vmm.h"

namespace pkv {
void set_last_error_message(const char* msg);
}

namespace {

struct Driver {
  PFN_cuMemAddressReserve_v10020 reserve = nullptr;
  PFN_cuMemAddressFree_v10020 addr_free = nullptr;
  PFN_cuMemCreate_v10020 create = nullptr;
  PFN_cuMemRelease_v10020 release = nullptr;
  PFN_cuMemMap_v10020 map = nullptr;
  PFN_cuMemUnmap_v10020 unmap = nullptr;
  PFN_cuMemSetAccess_v10020 set_access = nullptr;
  PFN_cuMemGetAllocationGranularity_v10020 granularity = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F* fn) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || f == nullptr)
    return false;
  *fn = reinterpret_cast<F>(f);
  return true;
}

const Driver& driver() {
  static Driver d;
  static std::once_flag once;
  std::call_once(once, [] {
    d.ok = entry("cuMemAddressReserve", &d.reserve) && entry("cuMemAddressFree", &d.addr_free) &&
           entry("cuMemCreate", &d.create) && entry("cuMemRelease", &d.release) &&
           entry("cuMemMap", &d.map) && entry("cuMemUnmap", &d.unmap) &&
           entry("cuMemSetAccess", &d.set_access) &&
           entry("cuMemGetAllocationGranularity", &d.granularity);
  });
  return d;
}

pkv_status vfail(pkv_status s, const char* msg) {
  pkv::set_last_error_message(msg);
  return s;
}

constexpr int64_t kRowBytes = 256;  // 128 bf16

}  // namespace

struct pkv_vmm_buffer {
  int device = 0;
  int32_t max_reqs = 0, hkv = 0;
  int64_t S = 0;
  size_t page = 0;          // mapping granularity
  size_t span = 0;          // reserved bytes per tensor (a multiple of page)
  CUdeviceptr base[2] = {0, 0};  // K, V
  std::vector<int32_t> users;    // per page: requests whose rows it backs
  std::vector<CUmemGenericAllocationHandle> handle[2];  // per page (0 = none)
  std::vector<CUmemGenericAllocationHandle> pool[2];    // unmapped handles for reuse
  std::vector<int64_t> rows;     // per request: rows of each head that are backed
  int64_t mapped_pages = 0, created_pages = 0, map_calls = 0;
  double map_seconds = 0.0;

  // pages that back rows [0, nrows) of every KV head of request r (sorted, unique)
  void pages_of(int32_t r, int64_t nrows, std::vector<int64_t>* out) const {
    out->clear();
    if (nrows <= 0) return;
    for (int32_t h = 0; h < hkv; ++h) {
      const int64_t start = ((static_cast<int64_t>(r) * hkv + h) * S) * kRowBytes;
      const int64_t end = start + nrows * kRowBytes;  // exclusive
      for (int64_t p = start / static_cast<int64_t>(page); p <= (end - 1) / static_cast<int64_t>(page);
           ++p)
        if (out->empty() || out->back() != p) out->push_back(p);
    }
    std::sort(out->begin(), out->end());
    out->erase(std::unique(out->begin(), out->end()), out->end());
  }
};

namespace {

pkv_status map_page(pkv_vmm_buffer* b, int64_t p) {
  const Driver& d = driver();
  CUmemAllocationProp prop = {};
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  prop.location.id = b->device;
  CUmemAccessDesc access = {};
  access.location = prop.location;
  access.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  for (int t = 0; t < 2; ++t) {
    const char* what = nullptr;
    CUmemGenericAllocationHandle h = 0;
    if (!b->pool[t].empty()) {
      h = b->pool[t].back();
      b->pool[t].pop_back();
    } else if (d.create(&h, b->page, &prop, 0) == CUDA_SUCCESS) {
      ++b->created_pages;
    } else {
      what = "cuMemCreate failed (out of device memory?)";
    }
    const CUdeviceptr at = b->base[t] + static_cast<CUdeviceptr>(p) * b->page;
    if (what == nullptr && d.map(at, b->page, 0, h, 0) != CUDA_SUCCESS) {
      b->pool[t].push_back(h);
      what = "cuMemMap failed";
    }
    if (what == nullptr && d.set_access(at, b->page, &access, 1) != CUDA_SUCCESS) {
      d.unmap(at, b->page);
      b->pool[t].push_back(h);
      what = "cuMemSetAccess failed";
    }
    if (what != nullptr) {
      if (t == 1) {  // undo the K half of this page
        d.unmap(b->base[0] + static_cast<CUdeviceptr>(p) * b->page, b->page);
        b->pool[0].push_back(b->handle[0][p]);
        b->handle[0][p] = 0;
      }
      return vfail(PKV_ERR_CUDA, what);
    }
    b->handle[t][p] = h;
  }
  ++b->mapped_pages;
  ++b->map_calls;
  return PKV_OK;
}

void unmap_page(pkv_vmm_buffer* b, int64_t p) {
  const Driver& d = driver();
  for (int t = 0; t < 2; ++t) {
    if (b->handle[t][p] == 0) continue;
    d.unmap(b->base[t] + static_cast<CUdeviceptr>(p) * b->page, b->page);
    b->pool[t].push_back(b->handle[t][p]);
    b->handle[t][p] = 0;
  }
  --b->mapped_pages;
}

}  // namespace

extern "C" {

pkv_status pkv_vmm_create(int32_t max_reqs, int32_t num_kv_heads, int64_t S,
                          pkv_vmm_buffer** out) {
  if (out == nullptr) return vfail(PKV_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  if (max_reqs <= 0 || num_kv_heads <= 0 || S <= 0 || S % 16 != 0)
    return vfail(PKV_ERR_INVALID_ARG, "max_reqs, num_kv_heads >= 1 and S a positive multiple of 16");
  const Driver& d = driver();
  if (!d.ok) return vfail(PKV_ERR_CUDA, "CUDA virtual memory management calls not found");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return vfail(PKV_ERR_CUDA, "no CUDA device");
  cudaFree(nullptr);  // make sure the device's primary context exists
  CUmemAllocationProp prop = {};
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  prop.location.id = dev;
  size_t page = 0;
  if (d.granularity(&page, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS || page == 0)
    return vfail(PKV_ERR_CUDA, "cuMemGetAllocationGranularity failed");
  pkv_vmm_buffer* b = new (std::nothrow) pkv_vmm_buffer();
  if (b == nullptr) return vfail(PKV_ERR_INVALID_ARG, "out of host memory");
  b->device = dev;
  b->max_reqs = max_reqs;
  b->hkv = num_kv_heads;
  b->S = S;
  b->page = page;
  const size_t bytes = static_cast<size_t>(max_reqs) * num_kv_heads * S * kRowBytes;
  b->span = (bytes + page - 1) / page * page;
  const size_t npages = b->span / page;
  for (int t = 0; t < 2; ++t) {
    if (d.reserve(&b->base[t], b->span, page, 0, 0) != CUDA_SUCCESS) {
      if (t == 1) d.addr_free(b->base[0], b->span);
      delete b;
      return vfail(PKV_ERR_CUDA, "cuMemAddressReserve failed");
    }
    b->handle[t].assign(npages, 0);
  }
  b->users.assign(npages, 0);
  b->rows.assign(max_reqs, 0);
  *out = b;
  return PKV_OK;
}

void* pkv_vmm_k(const pkv_vmm_buffer* b) { return b ? reinterpret_cast<void*>(b->base[0]) : nullptr; }
void* pkv_vmm_v(const pkv_vmm_buffer* b) { return b ? reinterpret_cast<void*>(b->base[1]) : nullptr; }

pkv_status pkv_vmm_ensure(pkv_vmm_buffer* b, int32_t req, int64_t tokens) {
  if (b == nullptr || req < 0 || req >= b->max_reqs || tokens < 0 || tokens > b->S)
    return vfail(PKV_ERR_INVALID_ARG, "bad request id or token count");
  const int64_t need = std::min<int64_t>((tokens + 15) / 16 * 16, b->S);  // whole 16-row tiles
  if (need <= b->rows[req]) return PKV_OK;
  const auto t0 = std::chrono::steady_clock::now();
  std::vector<int64_t> have, want;
  b->pages_of(req, b->rows[req], &have);
  b->pages_of(req, need, &want);
  std::vector<int64_t> added;
  std::set_difference(want.begin(), want.end(), have.begin(), have.end(), std::back_inserter(added));
  // map what no request has mapped yet, then count the new users
  std::vector<int64_t> fresh;
  for (int64_t p : added) {
    if (b->users[p] != 0) continue;
    const pkv_status st = map_page(b, p);
    if (st != PKV_OK) {
      for (int64_t q : fresh) unmap_page(b, q);  // nothing changed
      return st;
    }
    fresh.push_back(p);
  }
  for (int64_t p : added) ++b->users[p];
  b->rows[req] = need;
  b->map_seconds += std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  return PKV_OK;
}

pkv_status pkv_vmm_release(pkv_vmm_buffer* b, int32_t req) {
  if (b == nullptr || req < 0 || req >= b->max_reqs)
    return vfail(PKV_ERR_INVALID_ARG, "bad request id");
  // no kernel may still read or write the pages that are about to go
  if (cudaDeviceSynchronize() != cudaSuccess) return vfail(PKV_ERR_CUDA, "device synchronize failed");
  std::vector<int64_t> have;
  b->pages_of(req, b->rows[req], &have);
  for (int64_t p : have)
    if (--b->users[p] == 0) unmap_page(b, p);
  b->rows[req] = 0;
  return PKV_OK;
}

int64_t pkv_vmm_backed_tokens(const pkv_vmm_buffer* b, int32_t req) {
  if (b == nullptr || req < 0 || req >= b->max_reqs) return -1;
  return b->rows[req];
}

pkv_status pkv_vmm_stats(const pkv_vmm_buffer* b, size_t* page_bytes, int64_t* mapped_pages,
                         int64_t* created_pages, int64_t* map_calls, double* map_seconds) {
  if (b == nullptr) return vfail(PKV_ERR_INVALID_ARG, "null buffer");
  if (page_bytes) *page_bytes = b->page;
  if (mapped_pages) *mapped_pages = b->mapped_pages;
  if (created_pages) *created_pages = b->created_pages;
  if (map_calls) *map_calls = b->map_calls;
  if (map_seconds) *map_seconds = b->map_seconds;
  return PKV_OK;
}

void pkv_vmm_destroy(pkv_vmm_buffer* b) {
  if (b == nullptr) return;
  const Driver& d = driver();
  cudaDeviceSynchronize();
  for (size_t p = 0; p < b->users.size(); ++p)
    if (b->handle[0][p] != 0 || b->handle[1][p] != 0) unmap_page(b, static_cast<int64_t>(p));
  for (int t = 0; t < 2; ++t) {
    for (CUmemGenericAllocationHandle h : b->pool[t]) d.release(h);
    d.addr_free(b->base[t], b->span);
  }
  delete b;
}

}  // extern "C"
