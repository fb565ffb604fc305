// Serialised states: a versioned header + S + conv state, in host memory
// (stream-ordered copies, completion marker written last) and in files
// (checksum; the old file is removed before the new one is renamed into
// place, so that a path holds either the newest state or nothing).
#include "gdn.h"
#include "host.h"

#include <cerrno>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#define GDN_API extern "C" __attribute__((visibility("default")))

using namespace gdn_host;

namespace {

constexpr char kMagic[8] = {'G', 'D', 'N', 'S', 'T', 'A', 'T', 'E'};
constexpr uint32_t kVersion = 1, kHeaderBytes = 128;

struct Header {   // little-endian on both hosts (x86-64 and aarch64)
    char magic[8];
    uint32_t version, header_bytes;
    uint64_t tag;
    int32_t n_qk_heads, n_v_heads, d_k, d_v, grid_c, in_dtype;
    int64_t committed;
    uint64_t state_bytes, conv_bytes;
    uint64_t checksum;   // FNV-1a-style over the payload's 64-bit words; 0 = not computed
    uint64_t complete;   // completion marker, written after the payload
    uint8_t pad[kHeaderBytes - 88];
};
static_assert(sizeof(Header) == kHeaderBytes, "header layout");
static_assert(offsetof(Header, complete) == 80 && offsetof(Header, pad) == 88, "header layout");

uint64_t marker_of(uint64_t tag, int64_t committed) {
    const uint64_t m = tag ^ ((uint64_t)committed * 0x9E3779B97F4A7C15ull) ^ 0x434F4D504C455445ull;  // "COMPLETE"
    return m ? m : 1;
}

uint64_t payload_checksum(const unsigned char *p, size_t bytes) {
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i + 8 <= bytes; i += 8) {
        uint64_t w;
        std::memcpy(&w, p + i, 8);
        h = (h ^ w) * 1099511628211ull;
    }
    return h ? h : 1;
}

size_t state_bytes(const gdn_layer_desc *d) { return (size_t)d->n_v_heads * d->d_k * d->d_v * sizeof(float); }
size_t conv_bytes(const gdn_layer_desc *d) { return 3 * (size_t)channels(d) * in_elt(d); }

Header make_header(const gdn_layer_desc *d, const gdn_session *s) {
    Header h;
    std::memset(&h, 0, sizeof(h));
    std::memcpy(h.magic, kMagic, 8);
    h.version = kVersion;
    h.header_bytes = kHeaderBytes;
    h.tag = s->tag;
    h.n_qk_heads = d->n_qk_heads; h.n_v_heads = d->n_v_heads; h.d_k = d->d_k; h.d_v = d->d_v;
    h.grid_c = d->grid_c; h.in_dtype = d->in_dtype;
    h.committed = s->committed;
    h.state_bytes = state_bytes(d);
    h.conv_bytes = conv_bytes(d);
    return h;
}

// Everything a restore checks on the header, before it touches any device memory.
gdn_status check_header(const gdn_layer_desc *d, const Header &h, size_t blob_bytes) {
    if (std::memcmp(h.magic, kMagic, 8) != 0) return fail(GDN_ERR_STATE_MISMATCH, "not a serialised GDN state");
    if (h.version != kVersion || h.header_bytes != kHeaderBytes)
        return fail(GDN_ERR_STATE_MISMATCH, "state format version %u (header %u bytes) is not %u", h.version,
                    h.header_bytes, kVersion);
    if (h.tag != tag_of(d) || h.n_qk_heads != d->n_qk_heads || h.n_v_heads != d->n_v_heads || h.d_k != d->d_k ||
        h.d_v != d->d_v || h.grid_c != d->grid_c || h.in_dtype != d->in_dtype)
        return fail(GDN_ERR_STATE_MISMATCH, "state belongs to another layer description (tag %llx, expected %llx)",
                    (unsigned long long)h.tag, (unsigned long long)tag_of(d));
    if (h.state_bytes != state_bytes(d) || h.conv_bytes != conv_bytes(d) || h.committed < 0)
        return fail(GDN_ERR_STATE_MISMATCH, "state sizes or committed length do not fit the description");
    if (blob_bytes < kHeaderBytes + h.state_bytes + h.conv_bytes)
        return fail(GDN_ERR_STATE_MISMATCH, "blob of %zu bytes is shorter than its header says", blob_bytes);
    if (h.complete != marker_of(h.tag, h.committed))
        return fail(GDN_ERR_STATE_MISMATCH, "state is incomplete (its completion marker was never written)");
    return GDN_OK;
}

struct MarkerJob {
    volatile uint64_t *where;
    uint64_t value;
};
void CUDART_CB write_marker(void *p) {
    MarkerJob *j = static_cast<MarkerJob *>(p);
    __atomic_store_n(j->where, j->value, __ATOMIC_RELEASE);
    std::free(j);
}

struct PinnedBuffer {
    void *p = nullptr;
    ~PinnedBuffer() {
        if (p) cudaFreeHost(p);
    }
};

}  // namespace

GDN_API size_t gdn_state_blob_bytes(const gdn_layer_desc *d) {
    if (check_desc(d) != GDN_OK) return 0;
    return kHeaderBytes + state_bytes(d) + conv_bytes(d);
}

GDN_API gdn_status gdn_state_serialize(const gdn_layer_desc *d, const gdn_session *s, void *blob, size_t blob_bytes,
                                       gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if ((st = check_state(d, s, "session", true)) != GDN_OK) return st;
    if (!blob || blob_bytes < gdn_state_blob_bytes(d))
        return fail(GDN_ERR_INVALID_ARG, "blob needs %zu bytes", gdn_state_blob_bytes(d));
    if (reinterpret_cast<uintptr_t>(blob) & 7u) return fail(GDN_ERR_INVALID_ARG, "blob must be 8-byte aligned");
    MarkerJob *job = static_cast<MarkerJob *>(std::malloc(sizeof(MarkerJob)));
    if (!job) return fail(GDN_ERR_INVALID_ARG, "out of host memory");
    Header h = make_header(d, s);
    unsigned char *b = static_cast<unsigned char *>(blob);
    Header *hb = reinterpret_cast<Header *>(b);
    __atomic_store_n(&hb->complete, (uint64_t)0, __ATOMIC_RELEASE);   // the blob reads as missing from here on
    std::memcpy(b, &h, offsetof(Header, complete));
    std::memset(b + offsetof(Header, pad), 0, sizeof(h.pad));
    cudaStream_t cst = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(b + kHeaderBytes, s->S, h.state_bytes, cudaMemcpyDeviceToHost, cst);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(b + kHeaderBytes + h.state_bytes, s->conv, h.conv_bytes, cudaMemcpyDeviceToHost, cst);
    if (e == cudaSuccess) {
        job->where = &hb->complete;
        job->value = marker_of(h.tag, h.committed);
        e = cudaLaunchHostFunc(cst, write_marker, job);
    }
    if (e != cudaSuccess) {
        std::free(job);
        return cuda_fail(e, "state serialisation copies");
    }
    return GDN_OK;
}

GDN_API gdn_status gdn_state_deserialize(const gdn_layer_desc *d, const void *blob, size_t blob_bytes, gdn_session *dst,
                                         gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if (!blob || blob_bytes < kHeaderBytes) return fail(GDN_ERR_INVALID_ARG, "blob is NULL or shorter than a header");
    if ((st = check_state(d, dst, "destination session", false)) != GDN_OK) return st;
    Header h;
    std::memcpy(&h, blob, sizeof(h));
    h.complete = __atomic_load_n(&static_cast<const Header *>(blob)->complete, __ATOMIC_ACQUIRE);
    if ((st = check_header(d, h, blob_bytes)) != GDN_OK) return st;
    const unsigned char *b = static_cast<const unsigned char *>(blob);
    if (h.checksum && payload_checksum(b + kHeaderBytes, h.state_bytes + h.conv_bytes) != h.checksum)
        return fail(GDN_ERR_STATE_MISMATCH, "state payload does not match its checksum");
    cudaStream_t cst = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(dst->S, b + kHeaderBytes, h.state_bytes, cudaMemcpyHostToDevice, cst);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(dst->conv, b + kHeaderBytes + h.state_bytes, h.conv_bytes, cudaMemcpyHostToDevice, cst);
    if (e != cudaSuccess) return cuda_fail(e, "state restore copies");
    dst->committed = h.committed;
    dst->tag = h.tag;
    return GDN_OK;
}

namespace {

gdn_status io_fail(const char *what, const std::string &path) {
    return fail(GDN_ERR_IO, "%s %s: %s", what, path.c_str(), std::strerror(errno));
}

bool write_all(int fd, const unsigned char *p, size_t n) {
    while (n > 0) {
        const ssize_t w = ::write(fd, p, n);
        if (w < 0) {
            if (errno == EINTR) continue;
            return false;
        }
        p += w;
        n -= (size_t)w;
    }
    return true;
}

bool read_all(int fd, unsigned char *p, size_t n) {
    while (n > 0) {
        const ssize_t r = ::read(fd, p, n);
        if (r < 0) {
            if (errno == EINTR) continue;
            return false;
        }
        if (r == 0) return false;
        p += r;
        n -= (size_t)r;
    }
    return true;
}

std::string dir_of(const std::string &path) {
    const size_t k = path.find_last_of('/');
    return k == std::string::npos ? std::string(".") : (k == 0 ? std::string("/") : path.substr(0, k));
}

}  // namespace

GDN_API gdn_status gdn_state_save(const gdn_layer_desc *d, const gdn_session *s, const char *path, gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if ((st = check_state(d, s, "session", true)) != GDN_OK) return st;
    if (!path || !*path) return fail(GDN_ERR_INVALID_ARG, "path is empty");
    const std::string p(path), tmp = p + ".tmp";
    const size_t n = gdn_state_blob_bytes(d);
    PinnedBuffer buf;
    cudaError_t e = cudaMallocHost(&buf.p, n);
    if (e != cudaSuccess) return cuda_fail(e, "pinned staging buffer");
    // the old state goes first: from here on the path holds the new state or nothing
    if (::unlink(p.c_str()) != 0 && errno != ENOENT) return io_fail("cannot remove", p);
    if ((st = gdn_state_serialize(d, s, buf.p, n, stream)) != GDN_OK) return st;
    e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "state serialisation");
    unsigned char *b = static_cast<unsigned char *>(buf.p);
    Header *h = reinterpret_cast<Header *>(b);
    h->checksum = payload_checksum(b + kHeaderBytes, n - kHeaderBytes);
    const int fd = ::open(tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return io_fail("cannot create", tmp);
    const bool ok = write_all(fd, b, n) && ::fsync(fd) == 0;
    const int saved = errno;
    ::close(fd);
    if (!ok) {
        ::unlink(tmp.c_str());
        errno = saved;
        return io_fail("cannot write", tmp);
    }
    if (::rename(tmp.c_str(), p.c_str()) != 0) {
        const int r = errno;
        ::unlink(tmp.c_str());
        errno = r;
        return io_fail("cannot rename into", p);
    }
    const int dfd = ::open(dir_of(p).c_str(), O_RDONLY);
    if (dfd >= 0) {
        ::fsync(dfd);
        ::close(dfd);
    }
    return GDN_OK;
}

GDN_API gdn_status gdn_state_load(const gdn_layer_desc *d, const char *path, gdn_session *dst, gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if ((st = check_state(d, dst, "destination session", false)) != GDN_OK) return st;
    if (!path || !*path) return fail(GDN_ERR_INVALID_ARG, "path is empty");
    const std::string p(path);
    const int fd = ::open(p.c_str(), O_RDONLY);
    if (fd < 0) {
        if (errno == ENOENT) return fail(GDN_ERR_NOT_FOUND, "no saved state at %s", p.c_str());
        return io_fail("cannot open", p);
    }
    const size_t n = gdn_state_blob_bytes(d);
    struct stat sb;
    if (::fstat(fd, &sb) != 0) {
        const int r = errno;
        ::close(fd);
        errno = r;
        return io_fail("cannot stat", p);
    }
    if ((size_t)sb.st_size != n) {
        ::close(fd);
        return fail(GDN_ERR_STATE_MISMATCH, "%s holds %lld bytes, a state of this layer is %zu", p.c_str(),
                    (long long)sb.st_size, n);
    }
    std::vector<unsigned char> buf(n);   // pageable: the copies below finish before the call returns
    const bool ok = read_all(fd, buf.data(), n);
    const int r = errno;
    ::close(fd);
    if (!ok) {
        errno = r;
        return io_fail("cannot read", p);
    }
    Header h;
    std::memcpy(&h, buf.data(), sizeof(h));
    if (h.checksum == 0) return fail(GDN_ERR_STATE_MISMATCH, "%s carries no checksum", p.c_str());
    if ((st = gdn_state_deserialize(d, buf.data(), n, dst, stream)) != GDN_OK) return st;
    const cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "state load copies");
    return GDN_OK;
}
