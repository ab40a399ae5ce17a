// snapshot.cu -- cache snapshots: the K / V rows of a session and its span
// summaries, saved to and restored from a file.
//
// Superlinear release post (geeks.co.kr/post/2077), "why this matters": the
// point of fast long-context inference is to keep the cache rather than
// re-process the context, in memory for instant replies and on disk between
// sessions.  The summaries travel with the rows, so a restored session
// routes exactly as the saved one did.
//
// Host code only: the copies are cudaMemcpyAsync calls (one per chunk) on the
// caller's stream through a caller-owned staging buffer split in two halves,
// so that the device copy of one chunk overlaps the file I/O of the other.
#include <stdio.h>
#include <string.h>

#include "internal.h"

using namespace ssa;

namespace {

static_assert(sizeof(ssa_snapshot_header) == 64, "the header is 64 bytes");

size_t elem_bytes(int dtype) { return dtype == SSA_F32 ? 4 : 2; }

// One contiguous run of bytes on the device (a head's rows) and its place
// in the file's payload order.
struct Run {
  size_t dev_off;  // byte offset from the tensor base
  size_t bytes;
};

// The payload as (tensor, runs) in file order: K heads, V heads, summ heads.
struct Layout {
  int64_t n_tokens, n_summ;
  size_t kv_run, summ_run;       // bytes of one head's K (or V) rows, of its summaries
  size_t kv_head, summ_head;     // device head strides in bytes
  int64_t heads;
  uint64_t payload;
};

Layout make_layout(const Problem& pr, int64_t n_tokens) {
  Layout l;
  const size_t es = elem_bytes(pr.dtype);
  l.n_tokens = n_tokens;
  l.n_summ = n_tokens / pr.S;
  l.heads = (int64_t)pr.B * pr.Hkv;
  l.kv_run = (size_t)n_tokens * pr.d * es;
  l.summ_run = (size_t)l.n_summ * pr.d * 4;
  l.kv_head = (size_t)pr.L_cap * pr.d * es;
  l.summ_head = (size_t)pr.ns_cap * pr.d * 4;
  l.payload = (uint64_t)l.heads * (2 * l.kv_run + l.summ_run);
  return l;
}

// Chunks of every run of the three tensors, in file order, handed to fn(dev
// pointer, bytes).  Stops at the first failing status.
template <typename Fn>
int for_each_chunk(const Layout& l, uint8_t* K, uint8_t* V, uint8_t* summ, size_t chunk, Fn&& fn) {
  uint8_t* bases[3] = {K, V, summ};
  for (int t = 0; t < 3; ++t) {
    const size_t run = t < 2 ? l.kv_run : l.summ_run;
    const size_t stride = t < 2 ? l.kv_head : l.summ_head;
    for (int64_t h = 0; h < l.heads; ++h) {
      for (size_t off = 0; off < run; off += chunk) {
        const size_t n = run - off < chunk ? run - off : chunk;
        const int rc = fn(bases[t] + (size_t)h * stride + off, n);
        if (rc != SSA_OK) return rc;
      }
    }
  }
  return SSA_OK;
}

int check_header(const ssa_snapshot_header& h, long long file_bytes) {
  if (memcmp(h.magic, SSA_SNAPSHOT_MAGIC, 8) != 0 || h.version != SSA_SNAPSHOT_VERSION) return SSA_ERR_IO;
  for (int i = 0; i < 8; ++i)
    if (h.reserved[i]) return SSA_ERR_IO;
  if (h.dtype != SSA_F32 && h.dtype != SSA_BF16 && h.dtype != SSA_F16) return SSA_ERR_IO;
  if (h.B < 1 || h.Hkv < 1 || h.d < 1 || h.S < 1 || h.n_tokens < 0) return SSA_ERR_IO;
  if (h.n_summ != h.n_tokens / h.S) return SSA_ERR_IO;
  const double want = (double)h.B * h.Hkv *
                      (2.0 * (double)h.n_tokens * h.d * elem_bytes(h.dtype) + (double)h.n_summ * h.d * 4.0);
  if (want > 9.0e18 || (double)h.payload_bytes != want) return SSA_ERR_IO;
  if (file_bytes != (long long)(64 + h.payload_bytes)) return SSA_ERR_IO;
  return SSA_OK;
}

long long file_size(FILE* f) {
  if (fseeko(f, 0, SEEK_END) != 0) return -1;
  const long long n = (long long)ftello(f);
  if (fseeko(f, 0, SEEK_SET) != 0) return -1;
  return n;
}

// Two events mark the device copies of the two staging halves.
struct Events {
  cudaEvent_t e[2] = {nullptr, nullptr};
  bool ok = false;
  Events() {
    ok = cudaEventCreateWithFlags(&e[0], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&e[1], cudaEventDisableTiming) == cudaSuccess;
  }
  ~Events() {
    for (auto x : e)
      if (x) cudaEventDestroy(x);
  }
};

bool staging_ok(const Problem& pr, const void* staging, size_t bytes) {
  return staging && bytes >= 2 * (size_t)pr.d * 4;
}

// Half of the staging buffer, rounded down to whole 16-byte units.
size_t half_of(size_t bytes) { return (bytes / 2) & ~(size_t)15; }

}  // namespace

extern "C" {

SSA_API int ssa_snapshot_read_header(const char* path, ssa_snapshot_header* out) {
  if (!path) return SSA_ERR_INVALID_ARG;
  FILE* f = fopen(path, "rb");
  if (!f) return SSA_ERR_IO;
  ssa_snapshot_header h;
  const long long n = file_size(f);
  const bool got = n >= 64 && fread(&h, 64, 1, f) == 1;
  fclose(f);
  if (!got) return SSA_ERR_IO;
  const int rc = check_header(h, n);
  if (rc == SSA_OK && out) *out = h;
  return rc;
}

SSA_API int ssa_snapshot_save(const ssa_params* p, int64_t n_tokens, const void* K, const void* V,
                              const float* summ, const char* path, void* staging, size_t staging_bytes,
                              void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (!K || !V || !summ || !path || n_tokens < 0 || n_tokens > pr.L) return SSA_ERR_INVALID_ARG;
  if (!staging_ok(pr, staging, staging_bytes)) return SSA_ERR_INVALID_ARG;
  const Layout l = make_layout(pr, n_tokens);
  ssa_snapshot_header h;
  memset(&h, 0, sizeof(h));
  memcpy(h.magic, SSA_SNAPSHOT_MAGIC, 8);
  h.version = SSA_SNAPSHOT_VERSION;
  h.dtype = pr.dtype;
  h.B = pr.B;
  h.Hkv = pr.Hkv;
  h.d = pr.d;
  h.S = pr.S;
  h.n_tokens = n_tokens;
  h.n_summ = l.n_summ;
  h.payload_bytes = l.payload;

  Events ev;
  if (!ev.ok) return SSA_ERR_CUDA;
  FILE* f = fopen(path, "wb");
  if (!f) return SSA_ERR_IO;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t half = half_of(staging_bytes);
  uint8_t* buf[2] = {static_cast<uint8_t*>(staging), static_cast<uint8_t*>(staging) + half};
  size_t pending_bytes = 0;  // bytes of the chunk copied into buf[slot ^ 1], not yet written
  int slot = 0;
  rc = fwrite(&h, 64, 1, f) == 1 ? SSA_OK : SSA_ERR_IO;
  // write out the chunk waiting in buf[s]
  auto flush = [&](int s) -> int {
    if (!pending_bytes) return SSA_OK;
    if (cudaEventSynchronize(ev.e[s]) != cudaSuccess) return SSA_ERR_CUDA;
    if (fwrite(buf[s], 1, pending_bytes, f) != pending_bytes) return SSA_ERR_IO;
    pending_bytes = 0;
    return SSA_OK;
  };
  if (rc == SSA_OK)
    rc = for_each_chunk(l, (uint8_t*)K, (uint8_t*)V, (uint8_t*)summ, half, [&](uint8_t* src, size_t n) -> int {
      // buf[slot] was last written out by the flush of the previous round
      if (cudaMemcpyAsync(buf[slot], src, n, cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSA_ERR_CUDA;
      if (cudaEventRecord(ev.e[slot], st) != cudaSuccess) return SSA_ERR_CUDA;
      const int r = flush(slot ^ 1);
      pending_bytes = n;
      slot ^= 1;
      return r;
    });
  if (rc == SSA_OK) rc = flush(slot ^ 1);
  if (rc != SSA_OK) cudaStreamSynchronize(st);  // no copy may still target the staging buffer
  if (fclose(f) != 0 && rc == SSA_OK) rc = SSA_ERR_IO;
  return rc;
}

SSA_API int ssa_snapshot_load(const ssa_params* p, const char* path, void* K, void* V, float* summ,
                              int64_t* n_tokens, void* staging, size_t staging_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (!K || !V || !summ || !path) return SSA_ERR_INVALID_ARG;
  if (!staging_ok(pr, staging, staging_bytes)) return SSA_ERR_INVALID_ARG;
  ssa_snapshot_header h;
  FILE* f = fopen(path, "rb");
  if (!f) return SSA_ERR_IO;
  const long long fbytes = file_size(f);
  if (fbytes < 64 || fread(&h, 64, 1, f) != 1 || check_header(h, fbytes) != SSA_OK || h.dtype != pr.dtype ||
      h.B != pr.B || h.Hkv != pr.Hkv || h.d != pr.d || h.S != pr.S || h.n_tokens > pr.L_cap) {
    fclose(f);
    return SSA_ERR_IO;
  }
  const Layout l = make_layout(pr, h.n_tokens);
  Events ev;
  if (!ev.ok) {
    fclose(f);
    return SSA_ERR_CUDA;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t half = half_of(staging_bytes);
  uint8_t* buf[2] = {static_cast<uint8_t*>(staging), static_cast<uint8_t*>(staging) + half};
  bool used[2] = {false, false};
  int slot = 0;
  rc = for_each_chunk(l, (uint8_t*)K, (uint8_t*)V, (uint8_t*)summ, half, [&](uint8_t* dst, size_t n) -> int {
    // the previous copy out of buf[slot] must be done before it is refilled
    if (used[slot] && cudaEventSynchronize(ev.e[slot]) != cudaSuccess) return SSA_ERR_CUDA;
    if (fread(buf[slot], 1, n, f) != n) return SSA_ERR_IO;
    if (cudaMemcpyAsync(dst, buf[slot], n, cudaMemcpyHostToDevice, st) != cudaSuccess) return SSA_ERR_CUDA;
    if (cudaEventRecord(ev.e[slot], st) != cudaSuccess) return SSA_ERR_CUDA;
    used[slot] = true;
    slot ^= 1;
    return SSA_OK;
  });
  const cudaError_t se = cudaStreamSynchronize(st);
  fclose(f);
  if (rc == SSA_OK && se != cudaSuccess) rc = SSA_ERR_CUDA;
  if (rc == SSA_OK && n_tokens) *n_tokens = h.n_tokens;
  return rc;
}

}  // extern "C"
