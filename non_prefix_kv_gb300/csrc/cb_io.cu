// Storage tier of the chunk-KV store: byte ranges of a file read into (pinned) host memory
// by parallel positional reads, the "fetch KV from storage" step of layer-wise loading
// (CacheBlend explainer, 0h-n0.github.io/posts/paper-2312-03052, §Pipelining and load
// controller: T_load of a storage device).  Host code only.
#include <errno.h>
#include <fcntl.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <sys/types.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <thread>
#include <vector>

#include "../../include/cacheblend.h"

namespace {

thread_local char g_io_msg[256] = "";

int io_fail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_io_msg, sizeof(g_io_msg), fmt, ap);
  va_end(ap);
  return CB_ERR_IO;
}

// reads [off, off + n) of fd into dst; returns 0 or an errno value (-1: end of file)
int read_range(int fd, uint64_t off, char* dst, size_t n) {
  while (n > 0) {
    const ssize_t r = pread(fd, dst, n, (off_t)off);
    if (r < 0) {
      if (errno == EINTR) continue;
      return errno;
    }
    if (r == 0) return -1;
    dst += r;
    off += (uint64_t)r;
    n -= (size_t)r;
  }
  return 0;
}

}  // namespace

extern "C" {

const char* cb_io_error_message(void) { return g_io_msg; }

int cb_file_read(const char* path, uint64_t offset, void* dst_host, size_t bytes, int32_t n_threads) {
  if (!path || (bytes > 0 && !dst_host)) return io_fail("file_read: NULL argument");
  if (bytes == 0) return CB_OK;
  const int fd = open(path, O_RDONLY);
  if (fd < 0) return io_fail("open %s: %s", path, strerror(errno));
  // pieces of at least 4 MB, at most n_threads of them
  const size_t min_piece = size_t(4) << 20;
  int nt = std::max(1, std::min<int>(n_threads < 1 ? 1 : n_threads, (int)((bytes + min_piece - 1) / min_piece)));
  std::atomic<int> err{0};
  auto work = [&](int t) {
    const size_t lo = bytes * (size_t)t / (size_t)nt, hi = bytes * (size_t)(t + 1) / (size_t)nt;
    const int e = read_range(fd, offset + lo, static_cast<char*>(dst_host) + lo, hi - lo);
    if (e) {
      int z = 0;
      err.compare_exchange_strong(z, e);
    }
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nt; ++t) pool.emplace_back(work, t);
  work(0);
  for (auto& th : pool) th.join();
  close(fd);
  const int e = err.load();
  if (e == -1) return io_fail("read %s: end of file before %llu bytes at offset %llu", path,
                              (unsigned long long)bytes, (unsigned long long)offset);
  if (e) return io_fail("read %s: %s", path, strerror(e));
  return CB_OK;
}

}  // extern "C"
