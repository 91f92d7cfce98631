// lsc_store.cpp -- the snapshot store of liblsc (include/lsc_store.h): the disk
// tier of the prefix cache.  Blobs (state snapshots, K/V blocks) and entries
// are checksummed files written through a temporary name; an in-memory index
// keeps sizes, reference counts, pins and recency for make_room.
//
// Source: "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "SSD 前缀缓存的写入与读取"
// and "磁盘缓存的完整性校验与容量管理"; the file format and the readings of
// the page are stated in include/lsc_store.h.
#include <cuda_runtime.h>
#include <dirent.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <cerrno>
#include <cinttypes>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <unordered_map>
#include <vector>

#include "lsc.h"
#include "lsc_internal.h"
#include "lsc_store.h"

namespace {

// ---- CRC-32C, slicing by 8 (tables built from the reflected polynomial) ----
struct Crc32c {
  uint32_t t[8][256];
  Crc32c() {
    for (uint32_t i = 0; i < 256; ++i) {
      uint32_t c = i;
      for (int k = 0; k < 8; ++k) c = (c >> 1) ^ ((c & 1) ? 0x82F63B78u : 0u);
      t[0][i] = c;
    }
    for (uint32_t i = 0; i < 256; ++i)
      for (int s = 1; s < 8; ++s) t[s][i] = (t[s - 1][i] >> 8) ^ t[0][t[s - 1][i] & 0xff];
  }
  uint32_t operator()(const uint8_t *p, size_t n, uint32_t crc = 0) const {
    crc = ~crc;
    while (n && ((uintptr_t)p & 7)) {
      crc = (crc >> 8) ^ t[0][(crc ^ *p++) & 0xff];
      --n;
    }
    while (n >= 8) {
      uint64_t w;
      std::memcpy(&w, p, 8);
      w ^= crc;  // the low 32 bits of a little-endian word meet the running CRC
      crc = t[7][w & 0xff] ^ t[6][(w >> 8) & 0xff] ^ t[5][(w >> 16) & 0xff] ^ t[4][(w >> 24) & 0xff] ^
            t[3][(w >> 32) & 0xff] ^ t[2][(w >> 40) & 0xff] ^ t[1][(w >> 48) & 0xff] ^ t[0][w >> 56];
      p += 8;
      n -= 8;
    }
    while (n--) crc = (crc >> 8) ^ t[0][(crc ^ *p++) & 0xff];
    return ~crc;
  }
};
const Crc32c &crc() {
  static const Crc32c c;
  return c;
}

// ---- CRC-32C of a concatenation from the CRCs of its parts ----
// The CRC register is an affine function of the input bits, and joining two
// messages cancels the pre- and post-inversion, so
//   crc(A || B) = crc(A) * x^(8 |B|) + crc(B)   (mod P, over GF(2)),
// with polynomials in the reflected representation the table CRC uses: bit 31
// holds the coefficient of x^0, bit 0 that of x^31, and multiplying by x is
// one zero-input step of the register.
uint32_t gf2_mulmod(uint32_t a, uint32_t b) {
  uint32_t prod = 0, bxk = b;  // bxk = b * x^k
  for (int k = 0; k < 32; ++k) {
    if (a & (0x80000000u >> k)) prod ^= bxk;
    bxk = (bxk >> 1) ^ ((bxk & 1) ? 0x82F63B78u : 0u);
  }
  return prod;
}
uint32_t x_pow_8n(uint64_t n) {  // x^(8 n) mod P by repeated squaring
  uint32_t r = 0x80000000u, sq = 0x80000000u >> 8;  // x^0, x^8
  for (; n; n >>= 1) {
    if (n & 1) r = gf2_mulmod(r, sq);
    sq = gf2_mulmod(sq, sq);
  }
  return r;
}
uint32_t crc_join(uint32_t crc_a, uint32_t crc_b, uint64_t len_b) { return gf2_mulmod(crc_a, x_pow_8n(len_b)) ^ crc_b; }

// ---- parallel file I/O ([KP]: the disk tier reads with up to four threads) ----
constexpr int kIoThreads = 4;
constexpr int64_t kIoPart = 4 << 20;  // default part size: payloads below two parts stay on one thread

// The part size: LSC_STORE_IO_PART (bytes, a positive multiple of 4096) when
// set, else kIoPart.
int64_t io_part_from_env() {
  const char *e = getenv("LSC_STORE_IO_PART");
  if (!e) return kIoPart;
  const long long v = atoll(e);
  return v > 0 && v % 4096 == 0 ? (int64_t)v : kIoPart;
}

struct Part {
  int64_t off, len;
  uint32_t crc;
  bool ok;
};

// Splits [0, n) into up to kIoThreads contiguous parts of at least `part`
// bytes (4 KiB-aligned boundaries) and runs fn(part) for each, the first on
// the calling thread.
template <typename F>
std::vector<Part> run_parts(int64_t n, int64_t part, F fn) {
  int t = (int)std::min<int64_t>(kIoThreads, std::max<int64_t>(1, n / part));
  std::vector<Part> parts((size_t)t);
  for (int i = 0; i < t; ++i) {
    const int64_t a = (n * i / t) & ~(int64_t)4095, b = i + 1 == t ? n : (n * (i + 1) / t) & ~(int64_t)4095;
    parts[(size_t)i] = Part{a, b - a, 0, false};
  }
  std::vector<std::thread> th;
  for (int i = 1; i < t; ++i) {
    try {
      th.emplace_back([&fn, &parts, i] { fn(parts[(size_t)i]); });
    } catch (...) {  // no thread: run the part here
      fn(parts[(size_t)i]);
    }
  }
  fn(parts[0]);
  for (auto &x : th) x.join();
  return parts;
}

// The CRC of the parts in order, or false when a part failed.
bool joined_crc(const std::vector<Part> &parts, uint32_t *out) {
  uint32_t c = 0;
  for (size_t i = 0; i < parts.size(); ++i) {
    if (!parts[i].ok) return false;
    c = i == 0 ? parts[i].crc : crc_join(c, parts[i].crc, (uint64_t)parts[i].len);
  }
  *out = c;
  return true;
}

constexpr int kHeader = 64;
constexpr uint32_t kVersion = 1;
constexpr int32_t kEntryKind = 255;
const char kMagic[8] = {'L', 'S', 'C', 'S', 'N', 'A', 'P', '1'};

void put_le(uint8_t *p, uint64_t v, int n) {
  for (int i = 0; i < n; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint64_t get_le(const uint8_t *p, int n) {
  uint64_t v = 0;
  for (int i = 0; i < n; ++i) v |= (uint64_t)p[i] << (8 * i);
  return v;
}

void make_header(uint8_t *h, int32_t kind, uint64_t ns, uint64_t key, uint64_t nbytes) {
  std::memset(h, 0, kHeader);
  std::memcpy(h, kMagic, 8);
  put_le(h + 8, kVersion, 4);
  put_le(h + 12, (uint32_t)kind, 4);
  put_le(h + 16, ns, 8);
  put_le(h + 24, key, 8);
  put_le(h + 32, nbytes, 8);
  put_le(h + 60, crc()(h, 60), 4);
}

// header checks: magic, CRC, version, namespace, key; returns the payload size or -1
int64_t check_header(const uint8_t *h, uint64_t ns, uint64_t key, int32_t *kind) {
  if (std::memcmp(h, kMagic, 8) != 0) return -1;
  if (get_le(h + 60, 4) != crc()(h, 60)) return -1;
  if (get_le(h + 8, 4) != kVersion || get_le(h + 16, 8) != ns || get_le(h + 24, 8) != key) return -1;
  if (kind) *kind = (int32_t)get_le(h + 12, 4);
  return (int64_t)get_le(h + 32, 8);
}

bool read_all(int fd, void *p, size_t n) {
  uint8_t *c = (uint8_t *)p;
  while (n) {
    const ssize_t r = ::read(fd, c, n);
    if (r < 0) {
      if (errno == EINTR) continue;
      return false;
    }
    if (r == 0) return false;
    c += r;
    n -= (size_t)r;
  }
  return true;
}

bool pread_all(int fd, void *p, size_t n, int64_t at) {
  uint8_t *c = (uint8_t *)p;
  while (n) {
    const ssize_t r = ::pread(fd, c, n, (off_t)at);
    if (r < 0) {
      if (errno == EINTR) continue;
      return false;
    }
    if (r == 0) return false;
    c += r;
    at += r;
    n -= (size_t)r;
  }
  return true;
}

bool pwrite_all(int fd, const void *p, size_t n, int64_t at) {
  const uint8_t *c = (const uint8_t *)p;
  while (n) {
    const ssize_t w = ::pwrite(fd, c, n, (off_t)at);
    if (w < 0) {
      if (errno == EINTR) continue;
      return false;
    }
    c += w;
    at += w;
    n -= (size_t)w;
  }
  return true;
}

struct Blob {
  int64_t size;  // file bytes
  int32_t kind;
  int32_t refs;
};
struct Entry {
  std::vector<uint64_t> blobs;
  int32_t pins;
  uint64_t last;
};

}  // namespace

struct lsc_store {
  std::string dir;
  uint64_t ns = 0;
  int64_t quota = 0, used = 0;
  uint64_t clock = 0;
  std::unordered_map<uint64_t, Blob> blobs;
  std::unordered_map<uint64_t, Entry> entries;
  int64_t io_part = kIoPart;  // parallel I/O part size
  void *pinned = nullptr;  // host staging of save/load_state
  size_t pinned_bytes = 0;

  std::string path(const char *sub, uint64_t key) const {
    char name[40];
    std::snprintf(name, sizeof(name), "/%s/%016" PRIx64, sub, key);
    return dir + name;
  }

  // temporary file + CRCs + rename ([KP]: a failed write removes the temporary
  // file); a large payload is checksummed and written by up to four threads
  int write_file(const char *sub, uint64_t key, int32_t kind, const void *data, int64_t bytes) {
    const std::string tmp = path("tmp", key), fin = path(sub, key);
    uint8_t h[kHeader];
    make_header(h, kind, ns, key, (uint64_t)bytes);
    const int fd = ::open(tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return LSC_ERR_IO;
    const uint8_t *d = (const uint8_t *)data;
    const std::vector<Part> parts = run_parts(bytes, io_part, [fd, d](Part &pt) {
      pt.crc = crc()(d + pt.off, (size_t)pt.len);
      pt.ok = pwrite_all(fd, d + pt.off, (size_t)pt.len, kHeader + pt.off);
    });
    uint32_t pc = 0;
    uint8_t c[4];
    bool ok = joined_crc(parts, &pc);
    put_le(c, pc, 4);
    ok = ok && pwrite_all(fd, h, kHeader, 0) && pwrite_all(fd, c, 4, kHeader + bytes) && ::fsync(fd) == 0;
    if (::close(fd) != 0 || !ok || ::rename(tmp.c_str(), fin.c_str()) != 0) {
      ::unlink(tmp.c_str());
      return LSC_ERR_IO;
    }
    return LSC_OK;
  }

  void touch(Entry &e) { e.last = ++clock; }

  void unlink_blob(uint64_t key) {
    auto it = blobs.find(key);
    used -= it->second.size;
    ::unlink(path("b", key).c_str());
    blobs.erase(it);
  }

  // an entry leaves: its blobs lose a reference; returns its blob keys
  std::vector<uint64_t> drop_entry_index(uint64_t key) {
    auto it = entries.find(key);
    std::vector<uint64_t> bl = std::move(it->second.blobs);
    for (uint64_t b : bl) --blobs[b].refs;
    entries.erase(it);
    ::unlink(path("e", key).c_str());
    return bl;
  }

  // [KP] make_room: unreferenced blocks first, then unpinned entries least
  // recently used first; blocks other entries still reference stay
  bool make_room(int64_t need) {
    if (used + need <= quota) return true;
    std::vector<uint64_t> unref;
    for (auto &kv : blobs)
      if (kv.second.refs == 0) unref.push_back(kv.first);
    std::sort(unref.begin(), unref.end());
    for (uint64_t k : unref) {
      unlink_blob(k);
      if (used + need <= quota) return true;
    }
    while (used + need > quota) {
      uint64_t victim = 0, best = UINT64_MAX;
      bool found = false;
      for (auto &kv : entries)
        if (kv.second.pins == 0 && kv.second.last < best) {
          best = kv.second.last;
          victim = kv.first;
          found = true;
        }
      if (!found) return false;
      std::vector<uint64_t> bl = drop_entry_index(victim);
      std::sort(bl.begin(), bl.end());
      bl.erase(std::unique(bl.begin(), bl.end()), bl.end());
      for (uint64_t b : bl)
        if (blobs.count(b) && blobs[b].refs == 0) unlink_blob(b);
    }
    return true;
  }

  // [KP] drop_damaged: the file and every entry that depends on it
  void drop_damaged(uint64_t key) {
    std::vector<uint64_t> dep;
    for (auto &kv : entries)
      if (std::find(kv.second.blobs.begin(), kv.second.blobs.end(), key) != kv.second.blobs.end())
        dep.push_back(kv.first);
    for (uint64_t e : dep) drop_entry_index(e);
    unlink_blob(key);
  }

  bool ensure_pinned(size_t n) {
    if (pinned_bytes >= n) return true;
    if (pinned) cudaFreeHost(pinned);
    pinned = nullptr;
    pinned_bytes = 0;
    if (cudaMallocHost(&pinned, n) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    pinned_bytes = n;
    return true;
  }
};

namespace {

bool mkdir_p(const std::string &d) {
  if (::mkdir(d.c_str(), 0755) == 0 || errno == EEXIST) return true;
  return false;
}

// The conv and ssm views of every GDN layer of a pool (via the public views).
struct SlotViews {
  std::vector<uint8_t *> conv, ssm;
  std::vector<int64_t> conv_bytes, ssm_bytes;
  int64_t page = 0, total = 0;
};
int slot_views(lsc_pool *pool, int32_t slot, SlotViews *sv) {
  if (slot < 0 || slot >= lsc_pool_num_slots(pool)) return LSC_ERR_OUT_OF_RANGE;
  for (int32_t l = 0;; ++l) {
    lsc_layer_view v;
    const int rc = lsc_pool_layer_view(pool, l, &v);
    if (rc == LSC_ERR_OUT_OF_RANGE) break;
    if (rc == LSC_ERR_STATELESS_LAYER) continue;
    if (rc != LSC_OK) return rc;
    sv->page = v.page_bytes;
    sv->conv.push_back((uint8_t *)v.conv + (int64_t)slot * v.page_bytes);
    sv->ssm.push_back((uint8_t *)v.ssm + (int64_t)slot * v.page_bytes);
    sv->conv_bytes.push_back(v.conv_bytes);
    sv->ssm_bytes.push_back(v.ssm_bytes);
    sv->total += v.conv_bytes + v.ssm_bytes;
  }
  return LSC_OK;
}

}  // namespace

extern "C" {

int lsc_store_open(const char *dir, uint64_t ns, int64_t quota, lsc_store **out) {
  if (!dir || !out || quota < 0) return LSC_ERR_INVALID_ARG;
  *out = nullptr;
  lsc_store *s = new (std::nothrow) lsc_store();
  if (!s) return LSC_ERR_NO_MEMORY;
  try {
    // one subdirectory per namespace: stores of other models or layouts never
    // see (or remove) each other's files
    char sub[24];
    std::snprintf(sub, sizeof(sub), "/%016" PRIx64, ns);
    s->dir = std::string(dir) + sub;
    s->ns = ns;
    s->quota = quota;
    s->io_part = io_part_from_env();
    if (!mkdir_p(dir) || !mkdir_p(s->dir) || !mkdir_p(s->dir + "/b") || !mkdir_p(s->dir + "/e") ||
        !mkdir_p(s->dir + "/tmp")) {
      delete s;
      return LSC_ERR_IO;
    }
    // rebuild the index: blob headers, entries in full; damaged files go
    auto scan = [&](const char *sub, std::vector<uint64_t> *keys) {
      DIR *d = ::opendir((s->dir + "/" + sub).c_str());
      if (!d) return false;
      while (dirent *e = ::readdir(d)) {
        char *end = nullptr;
        const uint64_t k = std::strtoull(e->d_name, &end, 16);
        if (e->d_name[0] == '.' || !end || *end || std::strlen(e->d_name) != 16) continue;
        keys->push_back(k);
      }
      ::closedir(d);
      return true;
    };
    std::vector<uint64_t> bk, ek;
    if (!scan("b", &bk) || !scan("e", &ek)) {
      delete s;
      return LSC_ERR_IO;
    }
    for (uint64_t k : bk) {
      const std::string p = s->path("b", k);
      struct stat st;
      uint8_t h[kHeader];
      int32_t kind = 0;
      const int fd = ::open(p.c_str(), O_RDONLY);
      const bool ok = fd >= 0 && ::fstat(fd, &st) == 0 && read_all(fd, h, kHeader);
      if (fd >= 0) ::close(fd);
      const int64_t n = ok ? check_header(h, ns, k, &kind) : -1;
      if (n < 0 || st.st_size != kHeader + n + 4 || kind == kEntryKind) {
        ::unlink(p.c_str());
        continue;
      }
      s->blobs[k] = Blob{(int64_t)st.st_size, kind, 0};
      s->used += st.st_size;
    }
    std::sort(ek.begin(), ek.end());  // recency of a reopened store: key order
    for (uint64_t k : ek) {
      const std::string p = s->path("e", k);
      std::vector<uint8_t> raw;
      struct stat st;
      const int fd = ::open(p.c_str(), O_RDONLY);
      bool ok = fd >= 0 && ::fstat(fd, &st) == 0 && st.st_size >= kHeader + 4;
      if (ok) {
        raw.resize((size_t)st.st_size);
        ok = read_all(fd, raw.data(), raw.size());
      }
      if (fd >= 0) ::close(fd);
      int32_t kind = 0;
      const int64_t n = ok ? check_header(raw.data(), ns, k, &kind) : -1;
      ok = n >= 0 && kind == kEntryKind && (int64_t)raw.size() == kHeader + n + 4 && n % 8 == 0 &&
           get_le(raw.data() + kHeader + n, 4) == crc()(raw.data() + kHeader, (size_t)n);
      Entry e{{}, 0, 0};
      for (int64_t i = 0; ok && i < n / 8; ++i) {
        const uint64_t b = get_le(raw.data() + kHeader + 8 * i, 8);
        ok = s->blobs.count(b) > 0;
        e.blobs.push_back(b);
      }
      if (!ok) {
        ::unlink(p.c_str());
        continue;
      }
      for (uint64_t b : e.blobs) ++s->blobs[b].refs;
      s->touch(e);
      s->entries.emplace(k, std::move(e));
    }
  } catch (...) {
    delete s;
    return LSC_ERR_NO_MEMORY;
  }
  *out = s;
  return LSC_OK;
}

int lsc_store_close(lsc_store *s) {
  if (!s) return LSC_ERR_INVALID_ARG;
  if (s->pinned) cudaFreeHost(s->pinned);
  delete s;
  return LSC_OK;
}

int lsc_store_put_blob(lsc_store *s, uint64_t key, int32_t kind, const void *data, int64_t bytes) {
  if (!s || key == 0 || kind == kEntryKind || bytes < 0 || (bytes > 0 && !data)) return LSC_ERR_INVALID_ARG;
  if (s->blobs.count(key)) return LSC_ERR_INVALID_ARG;
  const int64_t size = kHeader + bytes + 4;
  if (!s->make_room(size)) return LSC_ERR_NO_SPACE;
  const int rc = s->write_file("b", key, kind, data, bytes);
  if (rc != LSC_OK) return rc;
  s->blobs[key] = Blob{size, kind, 0};
  s->used += size;
  return LSC_OK;
}

int lsc_store_blob_size(const lsc_store *s, uint64_t key, int64_t *bytes) {
  if (!s || !bytes) return LSC_ERR_INVALID_ARG;
  auto it = s->blobs.find(key);
  if (it == s->blobs.end()) return LSC_ERR_NOT_FOUND;
  *bytes = it->second.size - kHeader - 4;
  return LSC_OK;
}

int lsc_store_get_blob(lsc_store *s, uint64_t key, void *dst, int64_t cap, int64_t *bytes, int32_t *kind) {
  if (!s || !bytes || cap < 0) return LSC_ERR_INVALID_ARG;
  auto it = s->blobs.find(key);
  if (it == s->blobs.end()) return LSC_ERR_NOT_FOUND;
  const int64_t n = it->second.size - kHeader - 4;
  *bytes = n;
  if (cap < n || (n > 0 && !dst)) return LSC_ERR_INVALID_ARG;
  const int fd = ::open(s->path("b", key).c_str(), O_RDONLY);
  if (fd < 0) return LSC_ERR_IO;
  uint8_t h[kHeader], c[4];
  int32_t k = 0;
  struct stat st;
  bool ok = ::fstat(fd, &st) == 0 && pread_all(fd, h, kHeader, 0) && check_header(h, s->ns, key, &k) == n &&
            st.st_size == kHeader + n + 4 && pread_all(fd, c, 4, kHeader + n);
  if (ok) {  // the payload, by up to four reader threads, each checksumming its part
    uint8_t *d = (uint8_t *)dst;
    const std::vector<Part> parts = run_parts(n, s->io_part, [fd, d](Part &pt) {
      pt.ok = pread_all(fd, d + pt.off, (size_t)pt.len, kHeader + pt.off);
      if (pt.ok) pt.crc = crc()(d + pt.off, (size_t)pt.len);
    });
    uint32_t pc = 0;
    ok = joined_crc(parts, &pc) && get_le(c, 4) == pc;
  }
  ::close(fd);
  if (!ok) {
    s->drop_damaged(key);
    return LSC_ERR_CORRUPT;
  }
  if (kind) *kind = k;
  return LSC_OK;
}

int lsc_store_put_entry(lsc_store *s, uint64_t key, const uint64_t *blob_keys, int32_t n) {
  if (!s || key == 0 || n < 0 || (n > 0 && !blob_keys) || s->entries.count(key)) return LSC_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!s->blobs.count(blob_keys[i])) return LSC_ERR_INVALID_ARG;
  std::vector<uint8_t> pay((size_t)n * 8);
  for (int32_t i = 0; i < n; ++i) put_le(pay.data() + 8 * i, blob_keys[i], 8);
  const int rc = s->write_file("e", key, kEntryKind, pay.data(), (int64_t)pay.size());
  if (rc != LSC_OK) return rc;
  Entry e{std::vector<uint64_t>(blob_keys, blob_keys + n), 0, 0};
  for (uint64_t b : e.blobs) ++s->blobs[b].refs;
  s->touch(e);
  s->entries.emplace(key, std::move(e));
  return LSC_OK;
}

int lsc_store_get_entry(const lsc_store *s, uint64_t key, uint64_t *blob_keys, int32_t cap, int32_t *n) {
  if (!s || !n || cap < 0) return LSC_ERR_INVALID_ARG;
  auto it = s->entries.find(key);
  if (it == s->entries.end()) return LSC_ERR_NOT_FOUND;
  *n = (int32_t)it->second.blobs.size();
  for (int32_t i = 0; i < *n && i < cap; ++i) blob_keys[i] = it->second.blobs[i];
  return LSC_OK;
}

int lsc_store_drop_entry(lsc_store *s, uint64_t key) {
  if (!s) return LSC_ERR_INVALID_ARG;
  if (!s->entries.count(key)) return LSC_ERR_NOT_FOUND;
  s->drop_entry_index(key);
  return LSC_OK;
}

int lsc_store_pin(lsc_store *s, uint64_t key) {
  if (!s) return LSC_ERR_INVALID_ARG;
  auto it = s->entries.find(key);
  if (it == s->entries.end()) return LSC_ERR_NOT_FOUND;
  ++it->second.pins;
  s->touch(it->second);
  return LSC_OK;
}

int lsc_store_unpin(lsc_store *s, uint64_t key) {
  if (!s) return LSC_ERR_INVALID_ARG;
  auto it = s->entries.find(key);
  if (it == s->entries.end()) return LSC_ERR_NOT_FOUND;
  if (it->second.pins == 0) return LSC_ERR_INVALID_ARG;
  --it->second.pins;
  s->touch(it->second);
  return LSC_OK;
}

int lsc_store_stats_get(const lsc_store *s, lsc_store_stats *o) {
  if (!s || !o) return LSC_ERR_INVALID_ARG;
  std::memset(o, 0, sizeof(*o));
  o->used_bytes = s->used;
  o->quota_bytes = s->quota;
  o->n_blobs = (int32_t)s->blobs.size();
  o->n_entries = (int32_t)s->entries.size();
  for (auto &kv : s->blobs) o->n_unreferenced += kv.second.refs == 0;
  for (auto &kv : s->entries) o->n_pinned += kv.second.pins > 0;
  return LSC_OK;
}

int lsc_store_save_state(lsc_store *s, uint64_t key, lsc_pool *pool, int32_t slot, void *stream) {
  lsc::TraceRange trace_("lsc_store_save_state");
  if (!s || !pool) return LSC_ERR_INVALID_ARG;
  SlotViews sv;
  int rc = slot_views(pool, slot, &sv);
  if (rc != LSC_OK) return rc;
  if (key == 0 || s->blobs.count(key)) return LSC_ERR_INVALID_ARG;
  if (!s->ensure_pinned((size_t)std::max<int64_t>(sv.total, 1))) return LSC_ERR_NO_MEMORY;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *h = (uint8_t *)s->pinned;
  int64_t off = 0;
  for (size_t i = 0; i < sv.conv.size(); ++i) {
    if (cudaMemcpyAsync(h + off, sv.conv[i], (size_t)sv.conv_bytes[i], cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(h + off + sv.conv_bytes[i], sv.ssm[i], (size_t)sv.ssm_bytes[i], cudaMemcpyDeviceToHost,
                        st) != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_CUDA;
    }
    off += sv.conv_bytes[i] + sv.ssm_bytes[i];
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  return lsc_store_put_blob(s, key, 0, h, sv.total);
}

int lsc_store_load_state(lsc_store *s, uint64_t key, lsc_pool *pool, int32_t slot, void *stream) {
  lsc::TraceRange trace_("lsc_store_load_state");
  if (!s || !pool) return LSC_ERR_INVALID_ARG;
  SlotViews sv;
  int rc = slot_views(pool, slot, &sv);
  if (rc != LSC_OK) return rc;
  int64_t n = 0;
  rc = lsc_store_blob_size(s, key, &n);
  if (rc != LSC_OK) return rc;
  if (n != sv.total) return LSC_ERR_LAYOUT;
  if (!s->ensure_pinned((size_t)std::max<int64_t>(n, 1))) return LSC_ERR_NO_MEMORY;
  int32_t kind = -1;
  rc = lsc_store_get_blob(s, key, s->pinned, n, &n, &kind);
  if (rc != LSC_OK) return rc;
  if (kind != 0) return LSC_ERR_LAYOUT;
  cudaStream_t st = (cudaStream_t)stream;
  const uint8_t *h = (const uint8_t *)s->pinned;
  int64_t off = 0;
  for (size_t i = 0; i < sv.conv.size(); ++i) {
    if (cudaMemcpyAsync(sv.conv[i], h + off, (size_t)sv.conv_bytes[i], cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(sv.ssm[i], h + off + sv.conv_bytes[i], (size_t)sv.ssm_bytes[i], cudaMemcpyHostToDevice,
                        st) != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_CUDA;
    }
    off += sv.conv_bytes[i] + sv.ssm_bytes[i];
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  return LSC_OK;
}

}  // extern "C"
