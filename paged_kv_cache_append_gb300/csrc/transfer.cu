// transfer.cu -- host replicas of pool pages in the logical-order packed host
// layout, and the D2H / H2D copies between them and the device planes.
//
// "Paged KV cache" maintainer design page, host replica section: a host
// replica keeps no device page ids and no block-table holes; its pages are
// packed in logical order, each page holding the whole grouped payload of the
// typed pool, so an extent pays only for the pages it holds.  D2H / H2D
// transfers copy whole page payloads and may merge adjacent physical ids into
// fewer transfer runs.
//
// Packed page (this library's byte order within the page, innermost last):
//   for layer l, for plane i (K code, V code, K scale, V scale):
//     the H * 64 * row_bytes[i] bytes of page group g in plane (l, i),
// i.e. exactly the page-major device slice, so one run of consecutive page
// groups is one strided copy per (layer, plane).
#include <vector>

#include "internal.h"

using namespace nk;

namespace {

size_t page_payload(const nk_pool* p) {
  size_t b = 0;
  for (int i = 0; i < p->n_planes; ++i)
    b += p->plane[i].row_bytes * NK_PAGE_TOKENS * static_cast<size_t>(p->desc.num_kv_heads);
  return b * p->desc.num_layers;
}

// Runs of consecutive physical ids over the logical list: run r covers
// logical pages [first[r], first[r] + len[r]) with ids ids[first[r]] + k.
void make_runs(const int32_t* ids, int32_t n, std::vector<int32_t>& first, std::vector<int32_t>& len) {
  for (int32_t i = 0; i < n; ++i) {
    if (!first.empty() && ids[i] == ids[first.back()] + len.back()) {
      ++len.back();
    } else {
      first.push_back(i);
      len.push_back(1);
    }
  }
}

int copy_pages(const nk_pool* p, const int32_t* ids, int32_t n, char* host, bool to_host, cudaStream_t s) {
  if (!p || (!ids && n > 0) || (!host && n > 0)) return fail(NK_ERR_INVALID_ARG, "null argument");
  if (n < 0) return fail(NK_ERR_SHAPE, "page count must be >= 0");
  for (int32_t i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= p->M)
      return fail(NK_ERR_RANGE, "page id " + std::to_string(ids[i]) + " at logical page " +
                                    std::to_string(i) + " outside [0, M)");
  std::vector<int32_t> first, len;
  make_runs(ids, n, first, len);
  const size_t pb = page_payload(p);
  const int H = p->desc.num_kv_heads;
  const int hm = p->desc.order == NK_HEAD_MAJOR;
  for (size_t r = 0; r < first.size(); ++r) {
    const int g0 = ids[first[r]];
    size_t off = 0;  // byte offset of (layer, plane) inside a packed page
    for (int l = 0; l < p->desc.num_layers; ++l) {
      for (int i = 0; i < p->n_planes; ++i) {
        const size_t tile = p->plane[i].row_bytes * NK_PAGE_TOKENS;  // one (page, head) tile
        char* base = static_cast<char*>(p->ptrs[l * p->n_planes + i]);
        char* hst = host + static_cast<size_t>(first[r]) * pb + off;
        // page-major: the H tiles of a page are contiguous, and so are the pages
        // of a run (one copy); head-major: one copy per head, the run's pages
        // of that head are contiguous
        const int parts = hm ? H : 1;
        const size_t width = hm ? tile : tile * H;
        for (int hh = 0; hh < parts; ++hh) {
          char* dev = base + static_cast<size_t>(tile_row(g0, hh, H, p->M, hm)) * p->plane[i].row_bytes;
          char* hp = hst + hh * tile;
          cudaError_t e = to_host
              ? cudaMemcpy2DAsync(hp, pb, dev, width, width, len[r], cudaMemcpyDeviceToHost, s)
              : cudaMemcpy2DAsync(dev, width, hp, pb, width, len[r], cudaMemcpyHostToDevice, s);
          if (e != cudaSuccess) return cuda_fail(e, to_host ? "page run D2H" : "page run H2D");
        }
        off += tile * H;
      }
    }
  }
  return NK_OK;
}

}  // namespace

extern "C" int nk_host_page_bytes(const nk_pool* pool, size_t* bytes) {
  clear_error();
  if (!pool || !bytes) return fail(NK_ERR_INVALID_ARG, "null argument");
  *bytes = page_payload(pool);
  return NK_OK;
}

extern "C" int nk_page_runs(const int32_t* page_ids, int32_t n, int32_t* run_first, int32_t* run_len,
                            int32_t* n_runs) {
  clear_error();
  if ((!page_ids && n > 0) || !n_runs) return fail(NK_ERR_INVALID_ARG, "null argument");
  if (n < 0) return fail(NK_ERR_SHAPE, "page count must be >= 0");
  std::vector<int32_t> first, len;
  make_runs(page_ids, n, first, len);
  *n_runs = static_cast<int32_t>(first.size());
  for (size_t r = 0; r < first.size(); ++r) {
    if (run_first) run_first[r] = first[r];
    if (run_len) run_len[r] = len[r];
  }
  return NK_OK;
}

extern "C" int nk_pages_to_host(const nk_pool* pool, const int32_t* page_ids, int32_t n, void* host,
                                void* stream) {
  clear_error();
  return copy_pages(pool, page_ids, n, static_cast<char*>(host), true, static_cast<cudaStream_t>(stream));
}

extern "C" int nk_pages_from_host(nk_pool* pool, const int32_t* page_ids, int32_t n, const void* host,
                                  void* stream) {
  clear_error();
  return copy_pages(pool, page_ids, n, static_cast<char*>(const_cast<void*>(host)), false,
                    static_cast<cudaStream_t>(stream));
}
