// GGUF v3 reader: header, typed metadata, tensor-info table, 32-byte-aligned blob,
// and the copy of every payload to device memory, unchanged.
//
// Layout as given by "GGUF Inferencer in R" section 2.1 (byte blueprint) and
// "GGUF: The File Format Powering Local LLM Inference" ("What is stored inside a
// GGUF file", gguf_demo.py; "Worked example, step by step"):
//   "GGUF" | u32 version | u64 n_tensors | u64 n_kv
//   n_kv x  { string key | u32 value type | value }
//   n_tensors x { string name | u32 n_dims | n_dims x u64 extent | u32 type | u64 offset }
//   zero padding to a multiple of 32 | blob (tensor payloads at their offsets)
// Strings are u64 length + bytes (the lesson's reading; its worked example reaches
// data start 224 only with 8-byte lengths).  Unknown keys are stepped over by type.
#include <cerrno>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <new>

#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include "ggq_internal.h"

namespace ggq {

namespace {

constexpr uint64_t kAlign = 32;          // data blob alignment
constexpr uint64_t kArenaAlign = 256;    // device placement of each payload
constexpr int kMaxArrayDepth = 8;

// Bounds-checked little-endian cursor over the file bytes.
class Reader {
  public:
    Reader(const uint8_t* p, uint64_t n) : p_(p), n_(n) {}
    uint64_t pos() const { return pos_; }
    uint64_t left() const { return n_ - pos_; }
    bool u32(uint32_t* v) { return raw(v, 4); }
    bool u64(uint64_t* v) { return raw(v, 8); }
    bool skip(uint64_t k) {
        if (k > left()) return false;
        pos_ += k;
        return true;
    }
    bool str(std::string* s) {
        uint64_t len;
        if (!u64(&len) || len > left()) return false;
        s->assign(reinterpret_cast<const char*>(p_ + pos_), len);
        pos_ += len;
        return true;
    }
    const uint8_t* at(uint64_t off) const { return p_ + off; }

  private:
    bool raw(void* v, uint64_t k) {
        if (k > left()) return false;
        std::memcpy(v, p_ + pos_, k);  // the formats are little-endian, as are both hosts
        pos_ += k;
        return true;
    }
    const uint8_t* p_;
    uint64_t n_;
    uint64_t pos_ = 0;
};

// size in bytes of a fixed-size metadata scalar; 0 for string/array/unknown
uint64_t scalar_size(uint32_t t) {
    switch (t) {
    case GGQ_KV_U8: case GGQ_KV_I8: case GGQ_KV_BOOL: return 1;
    case GGQ_KV_U16: case GGQ_KV_I16: return 2;
    case GGQ_KV_U32: case GGQ_KV_I32: case GGQ_KV_F32: return 4;
    case GGQ_KV_U64: case GGQ_KV_I64: case GGQ_KV_F64: return 8;
    default: return 0;
    }
}

// Step over one value of type t; fails on truncation or an unknown type.
int skip_value(Reader& rd, uint32_t t, int depth) {
    if (uint64_t s = scalar_size(t)) {
        return rd.skip(s) ? GGQ_OK : fail(GGQ_EFORMAT, "metadata value truncated");
    }
    if (t == GGQ_KV_STRING) {
        uint64_t len;
        if (!rd.u64(&len) || !rd.skip(len)) return fail(GGQ_EFORMAT, "metadata string truncated");
        return GGQ_OK;
    }
    if (t == GGQ_KV_ARRAY) {
        if (depth >= kMaxArrayDepth) return fail(GGQ_EFORMAT, "metadata arrays nested too deep");
        uint32_t et;
        uint64_t count;
        if (!rd.u32(&et) || !rd.u64(&count)) return fail(GGQ_EFORMAT, "metadata array header truncated");
        if (uint64_t s = scalar_size(et)) {
            if (count > rd.left() / s) return fail(GGQ_EFORMAT, "metadata array runs past end of file");
            rd.skip(count * s);
            return GGQ_OK;
        }
        if (et != GGQ_KV_STRING && et != GGQ_KV_ARRAY)
            return fail(GGQ_EFORMAT, "unknown metadata array element type %u", et);
        // every string / array element takes at least 8 bytes
        if (count > rd.left() / 8) return fail(GGQ_EFORMAT, "metadata array runs past end of file");
        for (uint64_t i = 0; i < count; ++i) {
            int rc = skip_value(rd, et, depth + 1);
            if (rc) return rc;
        }
        return GGQ_OK;
    }
    return fail(GGQ_EFORMAT, "unknown metadata value type %u", t);
}

bool mul_ok(uint64_t a, uint64_t b, uint64_t* out) {
    if (a != 0 && b > UINT64_MAX / a) return false;
    *out = a * b;
    return true;
}

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

int parse(const uint8_t* buf, uint64_t len, ggq_model* m) {
    Reader rd(buf, len);
    if (len < 4 || std::memcmp(buf, "GGUF", 4) != 0) return fail(GGQ_EFORMAT, "bad magic (not a GGUF file)");
    rd.skip(4);
    uint64_t n_tensors, n_kv;
    if (!rd.u32(&m->version) || !rd.u64(&n_tensors) || !rd.u64(&n_kv))
        return fail(GGQ_EFORMAT, "header truncated");
    if (m->version != 3) return fail(GGQ_EFORMAT, "unsupported GGUF version %u (only 3)", m->version);
    // every KV takes >= 8+4+1 bytes and every tensor info >= 8+4+8+4+8
    if (n_kv > rd.left() / 13) return fail(GGQ_EFORMAT, "metadata count exceeds file size");
    if (n_tensors > rd.left() / 32) return fail(GGQ_EFORMAT, "tensor count exceeds file size");

    m->kvs.resize(n_kv);
    for (uint64_t i = 0; i < n_kv; ++i) {
        ggq_model::KV& kv = m->kvs[i];
        uint32_t t;
        if (!rd.str(&kv.key) || !rd.u32(&t)) return fail(GGQ_EFORMAT, "metadata entry %llu truncated",
                                                         (unsigned long long)i);
        kv.vtype = (int32_t)t;
        uint64_t start = rd.pos();
        int rc = skip_value(rd, t, 0);
        if (rc) return rc;
        if (t == GGQ_KV_STRING) start += 8;  // keep the bytes, not the length prefix
        kv.value.assign(rd.at(start), rd.at(rd.pos()));
    }

    m->tensors.resize(n_tensors);
    for (uint64_t i = 0; i < n_tensors; ++i) {
        ggq_model::Tensor& t = m->tensors[i];
        uint32_t nd, type;
        if (!rd.str(&t.name) || !rd.u32(&nd)) return fail(GGQ_EFORMAT, "tensor info %llu truncated",
                                                         (unsigned long long)i);
        if (nd < 1 || nd > 4) return fail(GGQ_EFORMAT, "tensor '%s': n_dims %u outside 1..4", t.name.c_str(), nd);
        t.n_dims = (int32_t)nd;
        uint64_t n = 1;
        for (uint32_t d = 0; d < nd; ++d) {
            uint64_t e;
            if (!rd.u64(&e)) return fail(GGQ_EFORMAT, "tensor '%s' dims truncated", t.name.c_str());
            if (e > (uint64_t)INT64_MAX || !mul_ok(n, e, &n) || n > ((uint64_t)1 << 62))
                return fail(GGQ_EFORMAT, "tensor '%s': element count overflows", t.name.c_str());
            t.ne[d] = (int64_t)e;
        }
        if (!rd.u32(&type) || !rd.u64(&t.offset))
            return fail(GGQ_EFORMAT, "tensor '%s' info truncated", t.name.c_str());
        t.type = (int32_t)type;
        int rc = payload_bytes(t.type, (uint64_t)t.ne[0], n, &t.nbytes);
        if (rc == GGQ_ETYPE) return fail(GGQ_ETYPE, "tensor '%s': unsupported type id %u", t.name.c_str(), type);
        if (rc) return fail(GGQ_EFORMAT, "tensor '%s': extent not a multiple of the block size", t.name.c_str());
    }
    m->data_start = align_up(rd.pos(), kAlign);
    if (m->data_start > len && n_tensors > 0) return fail(GGQ_EFORMAT, "file ends before the data blob");
    const uint64_t blob = len >= m->data_start ? len - m->data_start : 0;
    uint64_t arena = 0;
    for (auto& t : m->tensors) {
        if (t.offset % kAlign) return fail(GGQ_EFORMAT, "tensor '%s': offset not a multiple of 32", t.name.c_str());
        if (t.offset > blob || t.nbytes > blob - t.offset)
            return fail(GGQ_EFORMAT, "tensor '%s': payload runs past end of file", t.name.c_str());
        t.arena_off = arena;
        arena = align_up(arena + t.nbytes, kArenaAlign);
    }
    m->arena_bytes = arena;
    return GGQ_OK;
}

// Copy payloads to the device through two pinned staging buffers (overlapped).
int upload(const uint8_t* buf, ggq_model* m) {
    cudaError_t e = cudaGetDevice(&m->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (m->arena_bytes == 0) return GGQ_OK;
    e = cudaMalloc(&m->arena, m->arena_bytes);
    if (e == cudaErrorMemoryAllocation) {
        m->arena = nullptr;
        return fail(GGQ_ENOMEM, "cudaMalloc of %llu bytes failed", (unsigned long long)m->arena_bytes);
    }
    if (e != cudaSuccess) { m->arena = nullptr; return cuda_fail(e, "cudaMalloc"); }

    constexpr size_t kChunk = 32u << 20;
    void* stage[2] = {nullptr, nullptr};
    cudaStream_t s = nullptr;
    cudaEvent_t done[2] = {nullptr, nullptr};
    int rc = GGQ_OK;
    auto check = [&](cudaError_t err, const char* what) {
        if (err != cudaSuccess && rc == GGQ_OK) rc = cuda_fail(err, what);
        return rc == GGQ_OK;
    };
    if (check(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking), "cudaStreamCreate") &&
        check(cudaHostAlloc(&stage[0], kChunk, cudaHostAllocDefault), "cudaHostAlloc") &&
        check(cudaHostAlloc(&stage[1], kChunk, cudaHostAllocDefault), "cudaHostAlloc") &&
        check(cudaEventCreateWithFlags(&done[0], cudaEventDisableTiming), "cudaEventCreate") &&
        check(cudaEventCreateWithFlags(&done[1], cudaEventDisableTiming), "cudaEventCreate")) {
        int slot = 0;
        bool used[2] = {false, false};
        for (auto& t : m->tensors) {
            const uint8_t* src = buf + m->data_start + t.offset;
            uint8_t* dst = static_cast<uint8_t*>(m->arena) + t.arena_off;
            for (uint64_t off = 0; off < t.nbytes && rc == GGQ_OK; off += kChunk) {
                size_t n = (size_t)std::min<uint64_t>(kChunk, t.nbytes - off);
                if (used[slot] && !check(cudaEventSynchronize(done[slot]), "cudaEventSynchronize")) break;
                std::memcpy(stage[slot], src + off, n);
                if (!check(cudaMemcpyAsync(dst + off, stage[slot], n, cudaMemcpyHostToDevice, s),
                           "cudaMemcpyAsync") ||
                    !check(cudaEventRecord(done[slot], s), "cudaEventRecord"))
                    break;
                used[slot] = true;
                slot ^= 1;
            }
            if (rc) break;
        }
        check(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    }
    for (int i = 0; i < 2; ++i) {
        if (done[i]) cudaEventDestroy(done[i]);
        if (stage[i]) cudaFreeHost(stage[i]);
    }
    if (s) cudaStreamDestroy(s);
    return rc;
}

}  // namespace

int payload_bytes(int32_t type, uint64_t ne0, uint64_t n, uint64_t* out) {
    uint64_t per = 1, bytes = 0;
    switch (type) {
    case GGQ_F32: bytes = 4; break;
    case GGQ_F16: bytes = 2; break;
    // block sizes from "GGUF: The File Format Powering Local LLM Inference",
    // "What is quantization (in GGUF)" and its bits-per-weight table: an fp16
    // scale plus 32 one-byte codes (Q8_0) or 16 bytes of nibbles (Q4_0); 4.5
    // bits a weight for Q4_K and 6.5625 for Q6_K over 256-weight super-blocks
    case GGQ_Q4_0: per = 32; bytes = 18; break;
    case GGQ_Q8_0: per = 32; bytes = 34; break;
    case GGQ_Q4_K: per = 256; bytes = 144; break;
    case GGQ_Q6_K: per = 256; bytes = 210; break;
    default: *out = 0; return GGQ_ETYPE;
    }
    if (ne0 % per) { *out = 0; return GGQ_EFORMAT; }
    *out = n / per * bytes;
    return GGQ_OK;
}

}  // namespace ggq

using namespace ggq;

extern "C" int ggq_load_memory(const void* buf, size_t len, unsigned flags, ggq_model** out) {
    clear_error();
    if (!out) return fail(GGQ_EINVAL, "out is NULL");
    *out = nullptr;
    if (!buf && len) return fail(GGQ_EINVAL, "buf is NULL");
    std::unique_ptr<ggq_model> m(new (std::nothrow) ggq_model());
    if (!m) return fail(GGQ_ENOMEM, "host allocation failed");
    int rc;
    try {
        rc = parse(static_cast<const uint8_t*>(buf), len, m.get());
    } catch (const std::bad_alloc&) {
        return fail(GGQ_ENOMEM, "host allocation failed while parsing");
    }
    if (rc) return rc;
    if (!(flags & GGQ_LOAD_METADATA_ONLY)) {
        rc = upload(static_cast<const uint8_t*>(buf), m.get());
        if (rc) {
            if (m->arena) cudaFree(m->arena);
            return rc;
        }
    }
    *out = m.release();
    return GGQ_OK;
}

extern "C" int ggq_load_ex(const char* path, unsigned flags, ggq_model** out) {
    clear_error();
    if (!path || !out) return fail(GGQ_EINVAL, "NULL argument");
    *out = nullptr;
    int fd = open(path, O_RDONLY);
    if (fd < 0) return fail(GGQ_EIO, "cannot open '%s': %s", path, std::strerror(errno));
    struct stat st;
    if (fstat(fd, &st) != 0) {
        close(fd);
        return fail(GGQ_EIO, "cannot stat '%s'", path);
    }
    size_t len = (size_t)st.st_size;
    void* map = nullptr;
    if (len > 0) {
        map = mmap(nullptr, len, PROT_READ, MAP_PRIVATE, fd, 0);
        if (map == MAP_FAILED) {
            close(fd);
            return fail(GGQ_EIO, "cannot map '%s'", path);
        }
    }
    close(fd);
    int rc = ggq_load_memory(len ? map : "", len, flags, out);
    if (map) munmap(map, len);
    return rc;
}

extern "C" int ggq_load(const char* path, ggq_model** out) { return ggq_load_ex(path, 0, out); }

extern "C" void ggq_free(ggq_model* m) {
    if (!m) return;
    if (m->arena) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (m->device >= 0 && m->device != cur) cudaSetDevice(m->device);
        cudaFree(m->arena);
        if (cur >= 0 && m->device >= 0 && m->device != cur) cudaSetDevice(cur);
    }
    delete m;
}

extern "C" int ggq_version_of(const ggq_model* m, uint32_t* v) {
    if (!m || !v) return fail(GGQ_EINVAL, "NULL argument");
    *v = m->version;
    return GGQ_OK;
}

extern "C" int ggq_data_start(const ggq_model* m, uint64_t* off) {
    if (!m || !off) return fail(GGQ_EINVAL, "NULL argument");
    *off = m->data_start;
    return GGQ_OK;
}

extern "C" int ggq_num_tensors(const ggq_model* m, int64_t* n) {
    if (!m || !n) return fail(GGQ_EINVAL, "NULL argument");
    *n = (int64_t)m->tensors.size();
    return GGQ_OK;
}

extern "C" int ggq_tensor_info(const ggq_model* m, int64_t i, ggq_tensor* out) {
    if (!m || !out) return fail(GGQ_EINVAL, "NULL argument");
    if (i < 0 || (uint64_t)i >= m->tensors.size()) return fail(GGQ_EINVAL, "tensor index out of range");
    const auto& t = m->tensors[(size_t)i];
    out->name = t.name.c_str();
    out->type = t.type;
    out->n_dims = t.n_dims;
    for (int d = 0; d < 4; ++d) out->ne[d] = t.ne[d];
    out->offset = t.offset;
    out->nbytes = t.nbytes;
    out->data = m->arena ? static_cast<const uint8_t*>(m->arena) + t.arena_off : nullptr;
    return GGQ_OK;
}

extern "C" int ggq_find_tensor(const ggq_model* m, const char* name, int64_t* i) {
    if (!m || !name || !i) return fail(GGQ_EINVAL, "NULL argument");
    for (size_t k = 0; k < m->tensors.size(); ++k)
        if (m->tensors[k].name == name) { *i = (int64_t)k; return GGQ_OK; }
    return fail(GGQ_ENOTFOUND, "no tensor named '%s'", name);
}

extern "C" int ggq_num_kv(const ggq_model* m, int64_t* n) {
    if (!m || !n) return fail(GGQ_EINVAL, "NULL argument");
    *n = (int64_t)m->kvs.size();
    return GGQ_OK;
}

extern "C" int ggq_kv_info(const ggq_model* m, int64_t i, const char** key, int32_t* vtype,
                           const void** value, uint64_t* value_bytes) {
    if (!m) return fail(GGQ_EINVAL, "NULL argument");
    if (i < 0 || (uint64_t)i >= m->kvs.size()) return fail(GGQ_EINVAL, "metadata index out of range");
    const auto& kv = m->kvs[(size_t)i];
    if (key) *key = kv.key.c_str();
    if (vtype) *vtype = kv.vtype;
    if (value) *value = kv.value.data();
    if (value_bytes) *value_bytes = kv.value.size();
    return GGQ_OK;
}

extern "C" int ggq_kv_find(const ggq_model* m, const char* key, int64_t* i) {
    if (!m || !key || !i) return fail(GGQ_EINVAL, "NULL argument");
    for (size_t k = 0; k < m->kvs.size(); ++k)
        if (m->kvs[k].key == key) { *i = (int64_t)k; return GGQ_OK; }
    return fail(GGQ_ENOTFOUND, "no metadata key '%s'", key);
}
