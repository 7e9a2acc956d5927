// libpe: the C ABI and the host-side engine of the paged MoE layer.
//
// "Paged Experts" (SGLang docs), "The K-slot table and the host store": the
// GPU holds a K-row slot table per layer; a page-locked host store holds all
// E experts with exactly the slot layout, so a page-in is a plain row copy.
// The engine carves every device buffer out of one caller-owned arena (it
// never allocates device memory), owns the pinned host store, and turns a
// forward call into a fixed sequence of kernel launches on the caller's
// stream whose sizes depend only on shapes, which keeps it capturable in a
// CUDA graph ("Captured decode").

#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pe_internal.h"

using namespace pe;

namespace {

thread_local std::string g_create_error;

constexpr int kRouteInlineMaxTokens = 32;  // plan CTA routes up to one token per warp

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool dtype_ok(int d) {
    return d == PE_BF16 || d == PE_FP8_BLOCK128 || d == PE_INT4_GPTQ || d == PE_MXFP4 || d == PE_NVFP4;
}

bool is_fp4(int d) { return d == PE_MXFP4 || d == PE_NVFP4; }

// Expert width as the kernels see it.  MXFP4 and NVFP4 rows carry I padded
// to a multiple of 128 (zero codes, zero scales): the 4-bit kernels step
// through an expert's intermediate dimension in 128-input units, and the host
// row has exactly that padded layout, so what a page-in copies is what the
// kernels read.  Padded features contribute exact zeros.
int kernel_intermediate(const pe_config& c) {
    return is_fp4(c.dtype) ? (c.intermediate + 127) / 128 * 128 : c.intermediate;
}

// Returns "" when the config is valid, else the reason.
std::string validate(const pe_config& c) {
    if (c.num_layers < 1) return "num_layers must be >= 1";
    if (c.num_experts < 1 || c.num_experts > kMaxExperts) return "num_experts must be in 1..1024";
    if (c.top_k < 1 || c.top_k > kMaxTopK || c.top_k > c.num_experts) return "top_k must be in 1..min(E, 32)";
    if (c.num_slots < c.top_k) return "num_slots (K) must be >= top_k";
    if (c.num_slots > c.num_experts) return "num_slots (K) must be <= num_experts";
    if (c.hidden < 8 || c.hidden % 8) return "hidden must be a positive multiple of 8";
    if (c.intermediate < 8 || c.intermediate % 8) return "intermediate must be a positive multiple of 8";
    if (c.hidden > 16384 || c.intermediate > 16384) return "hidden/intermediate above 16384";
    if (c.max_tokens < 1) return "max_tokens must be >= 1";
    if (c.device < 0) return "device must be >= 0";
    if (c.dtype == PE_FP8_BLOCK128 && (c.hidden % kFp8Block || c.intermediate % kFp8Block))
        return "block-FP8 needs hidden and intermediate to be multiples of 128";
    if (c.dtype == PE_INT4_GPTQ && (c.hidden % kInt4Group || c.intermediate % kInt4Group))
        return "int4 needs hidden and intermediate to be multiples of the 128-input group";
    if (is_fp4(c.dtype) && c.hidden % 128)
        return "MXFP4 and NVFP4 need hidden to be a multiple of 128";
    if (c.dtype == PE_MXFP4 && c.intermediate % kMxfp4Block)
        return "MXFP4 needs intermediate to be a multiple of its 32-input block";
    if (c.dtype == PE_NVFP4 && c.intermediate % kNvfp4Block)
        return "NVFP4 needs intermediate to be a multiple of its 16-input block";
    return "";
}

void row_layout(const pe_config& c, pe_row_layout* r) {
    const uint64_t H = (uint64_t)c.hidden, I = (uint64_t)kernel_intermediate(c);
    std::memset(r, 0, sizeof(*r));
    // bytes per 2 weights: bf16 4, E4M3 2, 4-bit formats 1
    const uint64_t per2 = c.dtype == PE_BF16 ? 4 : c.dtype == PE_FP8_BLOCK128 ? 2 : 1;
    uint64_t s13 = 0, s2 = 0;
    if (c.dtype == PE_FP8_BLOCK128) {  // fp32 per 128x128 block
        s13 = 4 * ((2 * I + 127) / 128) * ((H + 127) / 128);
        s2 = 4 * ((H + 127) / 128) * ((I + 127) / 128);
    } else if (c.dtype == PE_INT4_GPTQ) {  // fp16 per output row and 128 inputs
        s13 = 2 * (2 * I) * ((H + kInt4Group - 1) / kInt4Group);
        s2 = 2 * H * ((I + kInt4Group - 1) / kInt4Group);
    } else if (is_fp4(c.dtype)) {  // one byte per row and block; NVFP4: a 16-byte fp32 tensor-scale header first
        const uint64_t blk = c.dtype == PE_MXFP4 ? kMxfp4Block : kNvfp4Block, hdr = c.dtype == PE_NVFP4 ? 16 : 0;
        s13 = hdr + (2 * I) * (H / blk);
        s2 = hdr + H * (I / blk);
    }
    r->w13_offset = 0;
    r->w13_bytes = I * H * per2;
    r->s13_offset = align_up(r->w13_offset + r->w13_bytes, 128);
    r->s13_bytes = s13;
    r->w2_offset = align_up(r->s13_offset + r->s13_bytes, 128);
    r->w2_bytes = H * I * per2 / 2;
    r->s2_offset = align_up(r->w2_offset + r->w2_bytes, 128);
    r->s2_bytes = s2;
    r->payload_bytes = r->w13_bytes + r->s13_bytes + r->w2_bytes + r->s2_bytes;
    r->row_stride = align_up(r->s2_offset + r->s2_bytes, 256);
}

Shape make_shape(const pe_config& c, const pe_row_layout& r) {
    Shape s;
    s.E = c.num_experts;
    s.k = c.top_k;
    s.K = c.num_slots;
    s.H = c.hidden;
    s.I = kernel_intermediate(c);
    s.Wmax = 1;
    s.dtype = c.dtype;
    s.stride = r.row_stride;
    s.copy_bytes = align_up(r.s2_offset + r.s2_bytes, 16);
    s.w13_off = r.w13_offset;
    s.s13_off = r.s13_offset;
    s.w2_off = r.w2_offset;
    s.s2_off = r.s2_offset;
    s.tail_off = r.s13_offset;
    return s;
}

// The tensor-core prefill path serves calls with more than kFusedMaxEntries
// entries when the shapes tile evenly.
bool tc_enabled(const pe_config& c, const pe_row_layout& r) {
    return (long long)c.max_tokens * c.top_k > kFusedMaxEntries && prefill_tc_supported(make_shape(c, r));
}

int32_t max_waves(const pe_config& c, int32_t T) {
    const long long ent = (long long)T * c.top_k;
    if (ent <= c.num_slots) return 1;
    const long long d = ent < c.num_experts ? ent : c.num_experts;
    return (int32_t)((d + c.num_slots - 1) / c.num_slots);
}

// Writes one MXFP4 / NVFP4 expert, given in its logical shape, into a host
// row of the padded layout: gate rows 0..I-1 and up rows I..2I-1 of w13 go
// to rows 0.. and Ip.. of the [2Ip, H/2] code block, each w2 row of I/2
// bytes to the start of an Ip/2-byte row, and the scale grids likewise (the
// NVFP4 tensor scale first, in the 16-byte header).  Everything else in the
// row is zero, so the padding the kernels read is the padding the row holds.
void load_fp4_row(const pe_config& c, const pe_row_layout& r, uint8_t* row, const uint8_t* w13, const uint8_t* w2,
                  const uint8_t* s13, const uint8_t* s2) {
    const size_t H = (size_t)c.hidden, I = (size_t)c.intermediate, Ip = (size_t)kernel_intermediate(c);
    const size_t blk = c.dtype == PE_MXFP4 ? kMxfp4Block : kNvfp4Block, hdr = c.dtype == PE_NVFP4 ? 16 : 0;
    std::memset(row, 0, r.row_stride);
    // w13 codes and scales: logical row j -> padded row j (gate) or Ip + j - I (up)
    const size_t cb = H / 2, sb = H / blk;
    for (size_t j = 0; j < 2 * I; ++j) {
        const size_t pj = j < I ? j : Ip + (j - I);
        std::memcpy(row + r.w13_offset + pj * cb, w13 + j * cb, cb);
        std::memcpy(row + r.s13_offset + hdr + pj * sb, s13 + hdr + j * sb, sb);
    }
    // w2 codes and scales: H rows, each I inputs wide inside Ip
    const size_t cw = I / 2, cwp = Ip / 2, sw = I / blk, swp = Ip / blk;
    for (size_t m = 0; m < H; ++m) {
        std::memcpy(row + r.w2_offset + m * cwp, w2 + m * cw, cw);
        std::memcpy(row + r.s2_offset + hdr + m * swp, s2 + hdr + m * sw, sw);
    }
    if (hdr) {  // the tensor scales
        std::memcpy(row + r.s13_offset, s13, 4);
        std::memcpy(row + r.s2_offset, s2, 4);
    }
}

// Bump allocator over the arena; with base == nullptr it only measures.
struct Carver {
    uint8_t* base;
    size_t off = 0;
    template <class T>
    T* take(size_t n) {
        off = align_up(off, 256);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += n * sizeof(T);
        return p;
    }
};

enum ProfKind {
    P_ROUTE = 0, P_PLAN, P_PAGEIN, P_GATEUP, P_GATEUP_PAGEIN, P_DOWN, P_SUM, P_ALIGN, P_PSTEP, P_DECODE, P_NUM
};
const char* kProfNames[P_NUM] = {"route",         "plan",     "pagein",        "gateup",
                                 "gateup_pagein", "down",     "topk_sum",      "prefill_align",
                                 "prefill_step",  "decode_step"};

}  // namespace

namespace pe {
void set_thread_error(const char* msg) { g_create_error = msg ? msg : ""; }
}  // namespace pe

struct pe_handle {
    pe_config cfg;
    pe_row_layout row;
    Shape shape;
    int maxTk = 0, Wmax = 0;
    uint8_t* slots = nullptr;
    uint8_t* store_host = nullptr;
    uint8_t* store_dev = nullptr;
    bool owns_store = false;      // the store was pinned by this handle (cudaHostAlloc)
    bool external_store = false;  // caller-owned memory registered by this handle (cudaHostRegister)
    std::vector<LayerDev> layers;
    uint8_t* loaded_dev = nullptr;   // [L][E]
    std::vector<uint8_t> loaded_host;
    uint32_t* err = nullptr;
    float* hbuf = nullptr;
    float* merged = nullptr;
    bool tc_ok = false;      // tensor-core prefill path available
    PrefillDev pre = {};
    PrefillMaps maps;
    int num_sms = 0;
    int decode_ctas_per_sm = 0;  // resident CTAs per SM of the decode step kernel (1 or 2)
    std::string last_error;
    // per-kernel timing
    bool prof_on = false;
    struct Mark { int kind; cudaEvent_t a, b; };
    std::vector<Mark> marks;
    std::vector<cudaEvent_t> pool;
    size_t pool_used = 0;
    double prof_ms[P_NUM] = {};
    uint64_t prof_n[P_NUM] = {};
};

namespace {

pe_status fail(pe_handle* h, pe_status st, const std::string& msg) {
    if (h)
        h->last_error = msg;
    else
        g_create_error = msg;
    return st;
}

pe_status cuda_fail(pe_handle* h, cudaError_t e, const char* what) {
    return fail(h, PE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

size_t carve(pe_handle* h, const pe_config& c, const pe_row_layout& r, uint8_t* base) {
    Carver cv{base};
    const int L = c.num_layers, E = c.num_experts, K = c.num_slots;
    const size_t maxTk = (size_t)c.max_tokens * c.top_k;
    const int W = max_waves(c, c.max_tokens);
    const bool tc = tc_enabled(c, r);
    // The prefill step pages an expert of a later wave into a staging row when
    // its slot is still in use, so the link need not wait: K rows right after
    // the slot table, so the weight tensor maps address them as slots.
    const int stage_rows = tc && W >= 2 ? K : 0;
    uint8_t* slots = cv.take<uint8_t>(((size_t)L * K + stage_rows) * r.row_stride);
    uint8_t* loaded = cv.take<uint8_t>((size_t)L * E);
    uint32_t* err = cv.take<uint32_t>(1);
    float* hbuf = cv.take<float>(maxTk * kernel_intermediate(c));
    float* merged = cv.take<float>(maxTk * c.hidden);
    PrefillDev pre = {};
    if (tc) {
        const size_t rows = prefill_max_rows((int)maxTk, E), tiles = prefill_max_tiles((int)maxTk, E);
        const size_t items = prefill_max_items(make_shape(c, r), tiles);
        pre.x_perm = cv.take<__nv_bfloat16>(rows * c.hidden);
        pre.h_perm = cv.take<__nv_bfloat16>(rows * kernel_intermediate(c));
        pre.perm = cv.take<int32_t>(rows);
        pre.tiles = cv.take<int4>(tiles);
        pre.items = cv.take<int2>(items);
        pre.members = cv.take<int4>(E);
        pre.pin_member = cv.take<int32_t>(E);
        pre.slot_need = cv.take<int32_t>(E);
        pre.landed = cv.take<unsigned>(E);
        pre.gu_done = cv.take<unsigned>(tiles);
        pre.slot_done = cv.take<unsigned>(K);
        pre.ctl = cv.take<unsigned>(4);
        pre.counts = cv.take<int32_t>(8);
        pre.stage_of = cv.take<int32_t>(E);
        pre.commit_member = cv.take<int32_t>(E);
        pre.stage_base = L * K;
        pre.stage_rows = stage_rows;
        pre.max_rows = (int)rows;
        pre.max_tiles = (int)tiles;
        pre.max_items = (int)items;
    }
    std::vector<LayerDev> layers(L);
    for (int l = 0; l < L; ++l) {
        LayerDev& d = layers[l];
        d.slot_expert = cv.take<int32_t>(K);
        d.slot_tick = cv.take<uint32_t>(K);
        d.expert_slot = cv.take<int32_t>(E);
        d.clock = cv.take<uint32_t>(1);
        d.counters = cv.take<unsigned long long>(C_NUM);
        d.plan_expert = cv.take<int32_t>((size_t)W * K);
        d.plan_slot = cv.take<int32_t>((size_t)W * K);
        d.plan_count = cv.take<int32_t>(W);
        d.member_expert = cv.take<int32_t>((size_t)W * K);
        d.member_slot = cv.take<int32_t>((size_t)W * K);
        d.member_count = cv.take<int32_t>(W);
        d.num_waves = cv.take<int32_t>(1);
        d.topk_id = cv.take<int32_t>(maxTk);
        d.topk_w = cv.take<float>(maxTk);
        d.entry_slot = cv.take<int32_t>(maxTk);
        d.entry_wave = cv.take<int32_t>(maxTk);
        d.loaded = loaded ? loaded + (size_t)l * E : nullptr;
        d.dsync = cv.take<unsigned>(16);
    }
    if (h) {
        h->slots = slots;
        h->loaded_dev = loaded;
        h->err = err;
        h->hbuf = hbuf;
        h->merged = merged;
        h->layers = layers;
        h->Wmax = W;
        h->maxTk = (int)maxTk;
        h->tc_ok = tc;
        h->pre = pre;
    }
    return align_up(cv.off, 256);
}

pe_status reset_state(pe_handle* h, cudaStream_t st) {
    const int E = h->cfg.num_experts, K = h->cfg.num_slots;
    for (auto& d : h->layers) {
        cudaError_t e = cudaMemsetAsync(d.slot_expert, 0xFF, sizeof(int32_t) * K, st);
        if (!e) e = cudaMemsetAsync(d.slot_tick, 0, sizeof(uint32_t) * K, st);
        if (!e) e = cudaMemsetAsync(d.expert_slot, 0xFF, sizeof(int32_t) * E, st);
        if (!e) e = cudaMemsetAsync(d.clock, 0, sizeof(uint32_t), st);
        if (!e) e = cudaMemsetAsync(d.dsync, 0, sizeof(unsigned) * 16, st);
        if (e) return cuda_fail(h, e, "reset residency");
    }
    return PE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tiled tensor map: bf16 with 128-byte swizzled boxes (inner box = 64
// elements), or unswizzled bytes (FP8 codes, decoded in shared memory).
bool encode_map(CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box, bool bytes) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
              const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16(CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* dims, const cuuint64_t* strides,
                 const cuuint32_t* box) {
    return encode_map(m, base, rank, dims, strides, box, false);
}

// Tensor maps over the prefill workspace and the whole slot table.
pe_status setup_prefill(pe_handle* h) {
    const pe_config& c = h->cfg;
    const PrefillDev& P = h->pre;
    const cuuint64_t H = (cuuint64_t)c.hidden, I = (cuuint64_t)kernel_intermediate(c), rows = (cuuint64_t)P.max_rows;
    const cuuint64_t nslots = (cuuint64_t)c.num_layers * c.num_slots + h->pre.stage_rows, stride = h->row.row_stride;
    bool ok = true;
    {
        const cuuint64_t d[2] = {H, rows}, st[1] = {H * 2};
        const cuuint32_t b[2] = {64, 128};
        ok = ok && encode_bf16(&h->maps.x_perm, P.x_perm, 2, d, st, b);
    }
    {
        const cuuint64_t d[2] = {I, rows}, st[1] = {I * 2};
        const cuuint32_t b[2] = {64, 128};
        ok = ok && encode_bf16(&h->maps.h_perm, P.h_perm, 2, d, st, b);
    }
    // weight boxes: BN/2 rows of w13 (the gate or the up half of a tile), BN rows of w2
    const cuuint32_t r13 = prefill_bn(c.dtype) / 2, r2 = prefill_bn(c.dtype);
    if (is_4bit(c.dtype)) {  // packed 4-bit code tiles (two codes per byte), decoded in shared memory
        {
            const cuuint64_t d[3] = {H / 2, 2 * I, nslots}, st[2] = {H / 2, stride};
            const cuuint32_t b[3] = {32, r13, 1};
            ok = ok && encode_map(&h->maps.w13, h->slots + h->row.w13_offset, 3, d, st, b, true);
        }
        {
            const cuuint64_t d[3] = {I / 2, H, nslots}, st[2] = {I / 2, stride};
            const cuuint32_t b[3] = {32, r2, 1};
            ok = ok && encode_map(&h->maps.w2, h->slots + h->row.w2_offset, 3, d, st, b, true);
        }
    } else if (c.dtype == PE_FP8_BLOCK128) {  // code tiles, decoded to bf16 in shared memory
        {
            const cuuint64_t d[3] = {H, 2 * I, nslots}, st[2] = {H, stride};
            const cuuint32_t b[3] = {64, r13, 1};
            ok = ok && encode_map(&h->maps.w13, h->slots + h->row.w13_offset, 3, d, st, b, true);
        }
        {
            const cuuint64_t d[3] = {I, H, nslots}, st[2] = {I, stride};
            const cuuint32_t b[3] = {64, r2, 1};
            ok = ok && encode_map(&h->maps.w2, h->slots + h->row.w2_offset, 3, d, st, b, true);
        }
    } else {
        {
            const cuuint64_t d[3] = {H, 2 * I, nslots}, st[2] = {H * 2, stride};
            const cuuint32_t b[3] = {64, r13, 1};
            ok = ok && encode_bf16(&h->maps.w13, h->slots + h->row.w13_offset, 3, d, st, b);
        }
        {
            const cuuint64_t d[3] = {I, H, nslots}, st[2] = {I * 2, stride};
            const cuuint32_t b[3] = {64, r2, 1};
            ok = ok && encode_bf16(&h->maps.w2, h->slots + h->row.w2_offset, 3, d, st, b);
        }
    }
    if (!ok) return fail(h, PE_ERR_CUDA, "could not encode the prefill tensor maps");
    cudaError_t e = prefill_setup_kernels();
    if (e) return cuda_fail(h, e, "prefill kernel attributes");
    return PE_OK;
}

// An external host store: caller-owned memory (for example one shared
// mapping that every replica process maps), registered for the handle's
// lifetime; `filled` marks every expert loaded.
struct ExternalStore {
    void* ptr = nullptr;
    size_t bytes = 0;
    int filled = 0;
};

// Registrations of external stores in this process, counted per start
// address: CUDA refuses to register a range twice, and several handles may
// share one store (a filling handle and reading handles, for instance).  The
// range is registered by its first handle and unregistered with its last.
std::mutex g_reg_mu;
std::vector<std::pair<void*, std::pair<size_t, int>>> g_regs;  // (ptr, (bytes, handles))

cudaError_t register_external(void* ptr, size_t bytes) {
    std::lock_guard<std::mutex> lock(g_reg_mu);
    for (auto& r : g_regs)
        if (r.first == ptr) {
            if (r.second.first < bytes) return cudaErrorInvalidValue;  // an overlapping, larger request
            r.second.second += 1;
            return cudaSuccess;
        }
    const cudaError_t e = cudaHostRegister(ptr, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (!e) g_regs.push_back({ptr, {bytes, 1}});
    return e;
}

void unregister_external(void* ptr) {
    std::lock_guard<std::mutex> lock(g_reg_mu);
    for (size_t i = 0; i < g_regs.size(); ++i)
        if (g_regs[i].first == ptr) {
            if (--g_regs[i].second.second == 0) {
                cudaHostUnregister(ptr);
                g_regs.erase(g_regs.begin() + (long)i);
            }
            return;
        }
}

pe_status create_impl(const pe_config* cfg, void* arena, size_t arena_bytes, pe_handle* owner,
                      const ExternalStore* ext, pe_handle** out) {
    if (!cfg || !out) return fail(nullptr, PE_ERR_INVALID, "NULL config or output pointer");
    *out = nullptr;
    if (!dtype_ok(cfg->dtype))
        return fail(nullptr, PE_ERR_UNSUPPORTED_DTYPE,
                    "expert dtype must be PE_BF16, PE_FP8_BLOCK128, PE_INT4_GPTQ, PE_MXFP4 or PE_NVFP4");
    const std::string why = validate(*cfg);
    if (!why.empty()) return fail(nullptr, PE_ERR_INVALID, why);
    if (owner) {
        const pe_config& o = owner->cfg;
        if (o.num_layers != cfg->num_layers || o.num_experts != cfg->num_experts ||
            o.hidden != cfg->hidden || o.intermediate != cfg->intermediate || o.dtype != cfg->dtype ||
            o.top_k != cfg->top_k || o.device != cfg->device)
            return fail(nullptr, PE_ERR_INVALID, "shared store needs the same L, E, top_k, H, I, dtype and device");
        if (!owner->owns_store && !owner->external_store)
            return fail(nullptr, PE_ERR_INVALID, "store owner must own or have registered its store");
    }
    if (ext) {  // checked before any CUDA call
        pe_row_layout rl;
        row_layout(*cfg, &rl);
        const size_t need = (size_t)cfg->num_layers * cfg->num_experts * rl.row_stride;
        if (!ext->ptr) return fail(nullptr, PE_ERR_INVALID, "external host store is NULL");
        if (reinterpret_cast<uintptr_t>(ext->ptr) % 4096)
            return fail(nullptr, PE_ERR_INVALID, "external host store must be 4096-byte aligned");
        if (ext->bytes < need)
            return fail(nullptr, PE_ERR_INVALID, "external host store too small: need " + std::to_string(need) + " bytes");
    }
    int ndev = 0;
    cudaError_t ce = cudaGetDeviceCount(&ndev);
    if (ce) return fail(nullptr, PE_ERR_CUDA, std::string("cudaGetDeviceCount: ") + cudaGetErrorString(ce));
    if (cfg->device >= ndev) return fail(nullptr, PE_ERR_INVALID, "device ordinal out of range");
    ce = cudaSetDevice(cfg->device);
    if (ce) return fail(nullptr, PE_ERR_CUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(ce));

    pe_row_layout r;
    row_layout(*cfg, &r);
    const size_t need = carve(nullptr, *cfg, r, nullptr);
    if (!arena) return fail(nullptr, PE_ERR_ARENA, "device arena is NULL");
    if (reinterpret_cast<uintptr_t>(arena) % 256) return fail(nullptr, PE_ERR_ARENA, "device arena must be 256-byte aligned");
    if (arena_bytes < need)
        return fail(nullptr, PE_ERR_ARENA, "device arena too small: need " + std::to_string(need) + " bytes");
    cudaPointerAttributes pa;
    ce = cudaPointerGetAttributes(&pa, arena);
    if (ce || pa.type != cudaMemoryTypeDevice || pa.device != cfg->device) {
        cudaGetLastError();
        return fail(nullptr, PE_ERR_ARENA, "device arena is not device memory of the configured device");
    }

    pe_handle* h = new pe_handle();
    h->cfg = *cfg;
    h->row = r;
    carve(h, *cfg, r, static_cast<uint8_t*>(arena));
    h->shape = make_shape(*cfg, r);
    h->shape.Wmax = h->Wmax;
    ce = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
    if (ce) {
        delete h;
        return fail(nullptr, PE_ERR_CUDA, std::string("device attribute: ") + cudaGetErrorString(ce));
    }
    ce = decode_setup_kernels();
    if (!ce) ce = decode_ctas_per_sm(cfg->dtype, &h->decode_ctas_per_sm);
    if (ce) {
        delete h;
        return fail(nullptr, PE_ERR_CUDA, std::string("decode kernel attributes: ") + cudaGetErrorString(ce));
    }
    // The one-kernel decode step and the prefill step order their phases
    // with counters that every CTA of the grid must reach, so all of a grid's
    // CTAs have to be resident at once; refuse a device where they cannot be.
    if (h->decode_ctas_per_sm < 1) {
        delete h;
        return fail(nullptr, PE_ERR_CUDA, "the decode step kernel cannot be resident on this device (occupancy 0)");
    }
    if (h->tc_ok && setup_prefill(h) != PE_OK) {
        const std::string msg = h->last_error;
        delete h;
        return fail(nullptr, PE_ERR_CUDA, msg);
    }
    if (h->tc_ok) {
        int n = 0;
        ce = prefill_step_ctas_per_sm(cfg->dtype, &n);
        if (ce || n < 1) {
            delete h;
            return fail(nullptr, PE_ERR_CUDA,
                        ce ? std::string("prefill occupancy: ") + cudaGetErrorString(ce)
                           : std::string("the prefill step kernel cannot be resident on this device (occupancy 0)"));
        }
    }

    const size_t store_bytes = (size_t)cfg->num_layers * cfg->num_experts * r.row_stride;
    if (owner) {
        h->store_host = owner->store_host;
        h->store_dev = owner->store_dev;
        h->owns_store = false;
        h->loaded_host = owner->loaded_host;
    } else if (ext) {
        ce = register_external(ext->ptr, store_bytes);
        if (ce) {
            cudaGetLastError();
            delete h;
            return fail(nullptr, PE_ERR_HOST_ALLOC,
                        std::string("could not register the external host store: ") + cudaGetErrorString(ce));
        }
        void* dp = nullptr;
        ce = cudaHostGetDevicePointer(&dp, ext->ptr, 0);
        if (ce) {
            unregister_external(ext->ptr);
            delete h;
            return fail(nullptr, PE_ERR_CUDA, std::string("cudaHostGetDevicePointer: ") + cudaGetErrorString(ce));
        }
        h->store_host = static_cast<uint8_t*>(ext->ptr);
        h->store_dev = static_cast<uint8_t*>(dp);
        h->external_store = true;
        h->loaded_host.assign((size_t)cfg->num_layers * cfg->num_experts, ext->filled ? 1 : 0);
    } else {
        void* p = nullptr;
        ce = cudaHostAlloc(&p, store_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
        if (ce || !p) {
            cudaGetLastError();
            delete h;
            return fail(nullptr, PE_ERR_HOST_ALLOC,
                        "could not pin a host store of " + std::to_string(store_bytes) + " bytes: " +
                            cudaGetErrorString(ce));
        }
        void* dp = nullptr;
        ce = cudaHostGetDevicePointer(&dp, p, 0);
        if (ce) {
            cudaFreeHost(p);
            delete h;
            return fail(nullptr, PE_ERR_CUDA, std::string("cudaHostGetDevicePointer: ") + cudaGetErrorString(ce));
        }
        h->store_host = static_cast<uint8_t*>(p);
        h->store_dev = static_cast<uint8_t*>(dp);
        h->owns_store = true;
        h->loaded_host.assign((size_t)cfg->num_layers * cfg->num_experts, 0);
    }
    // initial device state: every slot empty, counters and error word zero
    pe_status st = reset_state(h, nullptr);
    for (auto& d : h->layers)
        if (st == PE_OK && cudaMemset(d.counters, 0, sizeof(unsigned long long) * C_NUM)) st = PE_ERR_CUDA;
    if (st == PE_OK && cudaMemset(h->err, 0, sizeof(uint32_t))) st = PE_ERR_CUDA;
    if (st == PE_OK && cudaMemcpy(h->loaded_dev, h->loaded_host.data(), h->loaded_host.size(), cudaMemcpyHostToDevice))
        st = PE_ERR_CUDA;
    if (st == PE_OK && cudaDeviceSynchronize()) st = PE_ERR_CUDA;
    if (st != PE_OK) {
        const std::string msg = "device state init failed: " + h->last_error;
        if (h->owns_store) cudaFreeHost(h->store_host);
        if (h->external_store) unregister_external(h->store_host);
        delete h;
        return fail(nullptr, PE_ERR_CUDA, msg);
    }
    *out = h;
    return PE_OK;
}

// Per-kernel CUDA-event timing (profiling mode only).
cudaEvent_t take_event(pe_handle* h) {
    if (h->pool_used == h->pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e)) return nullptr;
        h->pool.push_back(e);
    }
    return h->pool[h->pool_used++];
}

void drain_marks(pe_handle* h) {
    for (auto& m : h->marks) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, m.a, m.b) == cudaSuccess) {
            h->prof_ms[m.kind] += ms;
            h->prof_n[m.kind] += 1;
        }
    }
    h->marks.clear();
    h->pool_used = 0;
}

struct ProfScope {
    pe_handle* h;
    int kind;
    cudaStream_t st;
    cudaEvent_t a = nullptr;
    ProfScope(pe_handle* h_, int k, cudaStream_t s) : h(h_), kind(k), st(s) {
        if (!h->prof_on) return;
        if (h->marks.size() >= 16384) {  // keep the event pool bounded
            cudaStreamSynchronize(st);
            drain_marks(h);
        }
        a = take_event(h);
        if (a) cudaEventRecord(a, st);
    }
    ~ProfScope() {
        if (!a) return;
        cudaEvent_t b = take_event(h);
        if (!b) return;
        cudaEventRecord(b, st);
        h->marks.push_back({kind, a, b});
    }
};

}  // namespace

extern "C" {

size_t pe_required_device_bytes(const pe_config* cfg) {
    if (!cfg || !dtype_ok(cfg->dtype) || !validate(*cfg).empty()) return 0;
    pe_row_layout r;
    row_layout(*cfg, &r);
    return carve(nullptr, *cfg, r, nullptr);
}

int32_t pe_slots_for_budget(const pe_config* cfg, size_t budget_bytes) {
    if (!cfg) return 0;
    pe_config c = *cfg;
    auto fits = [&](int32_t K) {
        c.num_slots = K;
        const size_t need = pe_required_device_bytes(&c);
        return need != 0 && need <= budget_bytes;
    };
    int32_t lo = cfg->top_k, hi = cfg->num_experts;  // the arena grows with K
    if (lo < 1 || hi < lo || !fits(lo)) return 0;
    while (lo < hi) {
        const int32_t mid = lo + (hi - lo + 1) / 2;
        if (fits(mid))
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

pe_status pe_get_row_layout(const pe_config* cfg, pe_row_layout* out) {
    if (!cfg || !out) return PE_ERR_INVALID;
    if (!dtype_ok(cfg->dtype)) return PE_ERR_UNSUPPORTED_DTYPE;
    if (!validate(*cfg).empty()) return PE_ERR_INVALID;
    row_layout(*cfg, out);
    return PE_OK;
}

int32_t pe_max_waves(const pe_config* cfg, int32_t num_tokens) {
    if (!cfg || num_tokens < 1 || !validate(*cfg).empty()) return 0;
    return max_waves(*cfg, num_tokens);
}

pe_status pe_create(const pe_config* cfg, void* dev_arena, size_t arena_bytes, pe_handle** out) {
    return create_impl(cfg, dev_arena, arena_bytes, nullptr, nullptr, out);
}

pe_status pe_create_external(const pe_config* cfg, void* dev_arena, size_t arena_bytes, void* host_store,
                             size_t host_store_bytes, int32_t filled, pe_handle** out) {
    ExternalStore ext;
    ext.ptr = host_store;
    ext.bytes = host_store_bytes;
    ext.filled = filled != 0;
    return create_impl(cfg, dev_arena, arena_bytes, nullptr, &ext, out);
}

pe_status pe_create_shared(const pe_config* cfg, void* dev_arena, size_t arena_bytes,
                           pe_handle* store_owner, pe_handle** out) {
    if (!store_owner) return fail(nullptr, PE_ERR_INVALID, "store_owner is NULL");
    return create_impl(cfg, dev_arena, arena_bytes, store_owner, nullptr, out);
}

pe_status pe_load_host_expert(pe_handle* h, int32_t layer, int32_t expert, const void* w13,
                              const void* w2, const void* s13, const void* s2) {
    if (!h) return PE_ERR_INVALID;
    if (!h->owns_store && !h->external_store)
        return fail(h, PE_ERR_INVALID, "load experts through the handle that owns or registered the host store");
    if (layer < 0 || layer >= h->cfg.num_layers || expert < 0 || expert >= h->cfg.num_experts)
        return fail(h, PE_ERR_RANGE, "layer or expert out of range");
    if (!w13 || !w2) return fail(h, PE_ERR_INVALID, "w13 and w2 must not be NULL");
    const bool scaled = h->cfg.dtype != PE_BF16;
    if (scaled && (!s13 || !s2)) return fail(h, PE_ERR_INVALID, "quantised experts need s13 and s2");
    if (!scaled && (s13 || s2)) return fail(h, PE_ERR_INVALID, "bf16 experts take no scales");
    const pe_row_layout& r = h->row;
    uint8_t* row = h->store_host + ((size_t)layer * h->cfg.num_experts + expert) * r.row_stride;
    if (is_fp4(h->cfg.dtype)) {
        load_fp4_row(h->cfg, r, row, static_cast<const uint8_t*>(w13), static_cast<const uint8_t*>(w2),
                     static_cast<const uint8_t*>(s13), static_cast<const uint8_t*>(s2));
    } else {
        std::memcpy(row + r.w13_offset, w13, r.w13_bytes);
        std::memcpy(row + r.w2_offset, w2, r.w2_bytes);
        if (scaled) {
            std::memcpy(row + r.s13_offset, s13, r.s13_bytes);
            std::memcpy(row + r.s2_offset, s2, r.s2_bytes);
        }
    }
    const size_t idx = (size_t)layer * h->cfg.num_experts + expert;
    if (!h->loaded_host[idx]) {
        h->loaded_host[idx] = 1;
        const uint8_t one = 1;
        cudaError_t e = cudaMemcpy(h->loaded_dev + idx, &one, 1, cudaMemcpyHostToDevice);
        if (e) return cuda_fail(h, e, "mark expert loaded");
    }
    return PE_OK;
}

void* pe_host_row(pe_handle* h, int32_t layer, int32_t expert) {
    if (!h || layer < 0 || layer >= h->cfg.num_layers || expert < 0 || expert >= h->cfg.num_experts)
        return nullptr;
    return h->store_host + ((size_t)layer * h->cfg.num_experts + expert) * h->row.row_stride;
}

pe_status pe_forward(pe_handle* h, int32_t layer, const void* hidden, const float* router_logits,
                     void* out, int32_t num_tokens, void* stream) {
    if (!h) return PE_ERR_INVALID;
    const pe_config& c = h->cfg;
    if (layer < 0 || layer >= c.num_layers) return fail(h, PE_ERR_RANGE, "layer out of range");
    if (num_tokens < 0 || num_tokens > c.max_tokens) return fail(h, PE_ERR_RANGE, "num_tokens outside 0..max_tokens");
    if (num_tokens == 0) return PE_OK;
    if (!hidden || !router_logits || !out) return fail(h, PE_ERR_INVALID, "NULL hidden, logits or out");
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(out)) % 16 ||
        reinterpret_cast<uintptr_t>(router_logits) % 4)
        return fail(h, PE_ERR_INVALID, "hidden/out must be 16-byte aligned, logits 4-byte aligned");
    if (hidden == out) return fail(h, PE_ERR_INVALID, "out may not alias hidden");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int T = num_tokens;
    const LayerDev& L = h->layers[layer];
    Shape s = h->shape;
    s.Wmax = max_waves(c, T);
    const size_t K = c.num_slots, E = c.num_experts;
    uint8_t* slots_layer = h->slots + (size_t)layer * K * s.stride;
    const uint8_t* host_layer = h->store_dev + (size_t)layer * E * s.stride;
    const auto* x = static_cast<const __nv_bfloat16*>(hidden);
    auto* y = static_cast<__nv_bfloat16*>(out);
    const int route_inline = T <= kRouteInlineMaxTokens;
    const int max_count = (int)((long long)T * c.top_k < (long long)K ? (long long)T * c.top_k : (long long)K);
    cudaError_t e = cudaSuccess;
    if (decode_fused_supported(s, T)) {
        // one wave of decode size: the whole step, plan included, in one kernel
        ProfScope p(h, P_DECODE, st);
        e = launch_decode_fused(L, s, router_logits, x, host_layer, slots_layer, T, h->hbuf, h->merged, y, L.dsync,
                                h->err, h->num_sms, h->decode_ctas_per_sm, st);
        if (e) return cuda_fail(h, e, "decode kernel");
        return PE_OK;
    }
    if (!route_inline) {
        ProfScope p(h, P_ROUTE, st);
        e = launch_route(L, s, router_logits, T, h->err, st);
        if (e) return cuda_fail(h, e, "route kernel");
    }
    {
        ProfScope p(h, P_PLAN, st);
        e = launch_plan(L, s, router_logits, T, route_inline, h->err, st);
        if (e) return cuda_fail(h, e, "plan kernel");
    }
    const int fused = s.Wmax == 1;
    // decode sizes page in inside the gate/up kernel; the choice depends on T
    // only, and both routes compute every h with the same code
    const bool pagein_fused = (long long)T * c.top_k <= kFusedMaxEntries;
    const int fmt = c.dtype;  // a pe_dtype
    if (!pagein_fused && h->tc_ok) {
        // prefill sizes: every wave's page-in and tensor-core GEMMs pipelined
        // in one kernel; every entry lands in the merged buffer, summed after
        {
            ProfScope p(h, P_ALIGN, st);
            e = launch_prefill_align(L, s, h->pre, x, layer * c.num_slots, T, h->num_sms, st);
            if (e) return cuda_fail(h, e, "prefill align kernels");
        }
        {
            ProfScope p(h, P_PSTEP, st);
            e = launch_prefill_step(L, s, h->pre, h->maps, host_layer, h->slots, layer * c.num_slots, h->merged,
                                    h->err, h->num_sms, st);
            if (e) return cuda_fail(h, e, "prefill step kernel");
        }
        ProfScope p(h, P_SUM, st);
        e = launch_topk_sum(s, h->merged, y, T, st);
        if (e) return cuda_fail(h, e, "top-k sum kernel");
        return PE_OK;
    }
    for (int w = 0; w < s.Wmax; ++w) {
        if (pagein_fused) {
            ProfScope p(h, P_GATEUP_PAGEIN, st);
            e = fmt == PE_FP8_BLOCK128
                    ? launch_gateup_pagein_fp8(L, s, x, host_layer, slots_layer, w, T, h->hbuf, h->num_sms, st)
                : is_4bit(fmt)
                    ? launch_gateup_pagein_q4(L, s, x, host_layer, slots_layer, w, T, h->hbuf, h->num_sms, st)
                    : launch_gateup_pagein(L, s, x, host_layer, slots_layer, w, T, h->hbuf, h->num_sms, st);
            if (e) return cuda_fail(h, e, "gate/up + page-in kernel");
        } else {
            {
                ProfScope p(h, P_PAGEIN, st);
                e = launch_pagein(L, s, host_layer, slots_layer, w, max_count, h->num_sms, st);
                if (e) return cuda_fail(h, e, "page-in kernel");
            }
            {
                ProfScope p(h, P_GATEUP, st);
                e = fmt == PE_FP8_BLOCK128 ? launch_gateup_fp8(L, s, x, slots_layer, w, T, h->hbuf, h->num_sms, st)
                    : is_4bit(fmt)         ? launch_gateup_q4(L, s, x, slots_layer, w, T, h->hbuf, h->num_sms, st)
                                           : launch_gateup(L, s, x, slots_layer, w, T, h->hbuf, h->num_sms, st);
                if (e) return cuda_fail(h, e, "gate/up kernel");
            }
        }
        {
            ProfScope p(h, P_DOWN, st);
            e = fmt == PE_FP8_BLOCK128
                    ? launch_down_fp8(L, s, slots_layer, w, T, h->hbuf, h->merged, y, fused, h->num_sms, st)
                : is_4bit(fmt)
                    ? launch_down_q4(L, s, slots_layer, w, T, h->hbuf, h->merged, y, fused, h->num_sms, st)
                    : launch_down(L, s, slots_layer, w, T, h->hbuf, h->merged, y, fused, h->num_sms, st);
            if (e) return cuda_fail(h, e, "down kernel");
        }
    }
    if (!fused) {
        ProfScope p(h, P_SUM, st);
        e = launch_topk_sum(s, h->merged, y, T, st);
        if (e) return cuda_fail(h, e, "top-k sum kernel");
    }
    return PE_OK;
}

pe_status pe_stats(pe_handle* h, int32_t layer, pe_stats_t* out) {
    if (!h || !out) return PE_ERR_INVALID;
    if (layer < -1 || layer >= h->cfg.num_layers) return fail(h, PE_ERR_RANGE, "layer out of range");
    cudaError_t e = cudaDeviceSynchronize();
    if (e) return cuda_fail(h, e, "synchronize");
    std::memset(out, 0, sizeof(*out));
    const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? h->cfg.num_layers : layer + 1;
    unsigned long long c[C_NUM];
    for (int l = l0; l < l1; ++l) {
        e = cudaMemcpy(c, h->layers[l].counters, sizeof(c), cudaMemcpyDeviceToHost);
        if (e) return cuda_fail(h, e, "read counters");
        out->steps += c[C_STEPS];
        out->waves += c[C_WAVES];
        out->entries += c[C_ENTRIES];
        out->distinct += c[C_DISTINCT];
        out->hits += c[C_HITS];
        out->page_ins += c[C_PAGE_INS];
        out->cold_fills += c[C_COLD];
    }
    out->bytes_paged = out->page_ins * h->row.payload_bytes;
    e = cudaMemcpy(&out->error_word, h->err, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e) return cuda_fail(h, e, "read error word");
    return PE_OK;
}

pe_status pe_read_plan(pe_handle* h, int32_t layer, int32_t num_tokens, pe_plan_view* out) {
    if (!h || !out) return PE_ERR_INVALID;
    if (layer < 0 || layer >= h->cfg.num_layers) return fail(h, PE_ERR_RANGE, "layer out of range");
    if (num_tokens < 1 || num_tokens > h->cfg.max_tokens) return fail(h, PE_ERR_RANGE, "num_tokens out of range");
    cudaError_t e = cudaDeviceSynchronize();
    if (e) return cuda_fail(h, e, "synchronize");
    const LayerDev& d = h->layers[layer];
    const size_t W = max_waves(h->cfg, num_tokens), K = h->cfg.num_slots;
    const size_t n = (size_t)num_tokens * h->cfg.top_k;
    struct Cp { void* dst; const void* src; size_t bytes; } cps[] = {
        {out->plan_expert, d.plan_expert, W * K * 4}, {out->plan_slot, d.plan_slot, W * K * 4},
        {out->plan_count, d.plan_count, W * 4},       {out->topk_id, d.topk_id, n * 4},
        {out->topk_w, d.topk_w, n * 4},               {out->entry_slot, d.entry_slot, n * 4},
        {out->entry_wave, d.entry_wave, n * 4},       {&out->num_waves, d.num_waves, 4}};
    for (auto& cp : cps) {
        if (!cp.dst) continue;
        e = cudaMemcpy(cp.dst, cp.src, cp.bytes, cudaMemcpyDeviceToHost);
        if (e) return cuda_fail(h, e, "read plan");
    }
    return PE_OK;
}

pe_status pe_read_residency(pe_handle* h, int32_t layer, int32_t* slot_expert, uint32_t* slot_tick,
                            int32_t* expert_slot, uint32_t* clock) {
    if (!h) return PE_ERR_INVALID;
    if (layer < 0 || layer >= h->cfg.num_layers) return fail(h, PE_ERR_RANGE, "layer out of range");
    cudaError_t e = cudaDeviceSynchronize();
    if (e) return cuda_fail(h, e, "synchronize");
    const LayerDev& d = h->layers[layer];
    const size_t K = h->cfg.num_slots, E = h->cfg.num_experts;
    if (slot_expert && (e = cudaMemcpy(slot_expert, d.slot_expert, 4 * K, cudaMemcpyDeviceToHost))) return cuda_fail(h, e, "read");
    if (slot_tick && (e = cudaMemcpy(slot_tick, d.slot_tick, 4 * K, cudaMemcpyDeviceToHost))) return cuda_fail(h, e, "read");
    if (expert_slot && (e = cudaMemcpy(expert_slot, d.expert_slot, 4 * E, cudaMemcpyDeviceToHost))) return cuda_fail(h, e, "read");
    if (clock && (e = cudaMemcpy(clock, d.clock, 4, cudaMemcpyDeviceToHost))) return cuda_fail(h, e, "read");
    return PE_OK;
}

pe_status pe_read_slot(pe_handle* h, int32_t layer, int32_t slot, void* host_dst, size_t bytes) {
    if (!h || !host_dst) return PE_ERR_INVALID;
    if (layer < 0 || layer >= h->cfg.num_layers || slot < 0 || slot >= h->cfg.num_slots || bytes > h->row.row_stride)
        return fail(h, PE_ERR_RANGE, "layer, slot or size out of range");
    cudaError_t e = cudaDeviceSynchronize();
    if (!e) e = cudaMemcpy(host_dst, h->slots + ((size_t)layer * h->cfg.num_slots + slot) * h->row.row_stride, bytes,
                           cudaMemcpyDeviceToHost);
    if (e) return cuda_fail(h, e, "read slot");
    return PE_OK;
}

pe_status pe_reset_residency(pe_handle* h, void* stream) {
    if (!h) return PE_ERR_INVALID;
    return reset_state(h, static_cast<cudaStream_t>(stream));
}

namespace {
// Words of the bounded-wait self-test: a word nothing ever sets, the abort
// word, and one error word per wait kind.
__device__ unsigned g_selftest_words[8];
}  // namespace

pe_status pe_selftest_bounded_waits(uint32_t poll_limit, uint32_t* out3) {
    if (!out3 || poll_limit == 0) return fail(nullptr, PE_ERR_INVALID, "out3 must not be NULL and poll_limit > 0");
    unsigned* w = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&w), g_selftest_words);
    if (!e) e = cudaMemset(w, 0, sizeof(unsigned) * 8);
    // w[0]: never set; w[1]: abort word; w[2..4]: error words
    if (!e) e = selftest_prefill_waits(w, w + 1, w + 2, w + 3, poll_limit, 0);
    if (!e) e = selftest_decode_wait(w, w + 4, poll_limit, 0);
    if (!e) e = cudaDeviceSynchronize();
    unsigned host[8] = {};
    if (!e) e = cudaMemcpy(host, w, sizeof(host), cudaMemcpyDeviceToHost);
    if (e) return fail(nullptr, PE_ERR_CUDA, std::string("bounded-wait self-test: ") + cudaGetErrorString(e));
    out3[0] = host[2];  // prefill step counter wait
    out3[1] = host[3];  // mbarrier wait
    out3[2] = host[4];  // decode step phase wait
    if (host[1] != 1u) out3[0] |= 0x80000000u;  // the abort word must have been raised
    return PE_OK;
}

pe_status pe_probe_host_link(pe_handle* h, void* dev_dst, size_t bytes, int32_t iters, void* stream,
                             double* copy_engine_gbs, double* kernel_gbs) {
    if (!h || !dev_dst || iters < 1) return PE_ERR_INVALID;
    const size_t store = (size_t)h->cfg.num_layers * h->cfg.num_experts * h->row.row_stride;
    bytes = (bytes < store ? bytes : store) / 16 * 16;
    if (bytes == 0) return fail(h, PE_ERR_INVALID, "probe size is zero");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t a, b;
    if (cudaEventCreate(&a)) return fail(h, PE_ERR_CUDA, "event");
    if (cudaEventCreate(&b)) { cudaEventDestroy(a); return fail(h, PE_ERR_CUDA, "event"); }
    cudaError_t e = cudaSuccess;
    float ms = 0.f;
    // warm-up of both paths
    e = cudaMemcpyAsync(dev_dst, h->store_host, bytes, cudaMemcpyHostToDevice, st);
    if (!e) e = launch_copy(h->store_dev, dev_dst, bytes, h->num_sms, st);
    if (!e) e = cudaEventRecord(a, st);
    for (int i = 0; !e && i < iters; ++i) e = cudaMemcpyAsync(dev_dst, h->store_host, bytes, cudaMemcpyHostToDevice, st);
    if (!e) e = cudaEventRecord(b, st);
    if (!e) e = cudaEventSynchronize(b);
    if (!e) e = cudaEventElapsedTime(&ms, a, b);
    if (!e && copy_engine_gbs) *copy_engine_gbs = (double)bytes * iters / (ms * 1e-3) / 1e9;
    if (!e) e = cudaEventRecord(a, st);
    for (int i = 0; !e && i < iters; ++i) e = launch_copy(h->store_dev, dev_dst, bytes, h->num_sms, st);
    if (!e) e = cudaEventRecord(b, st);
    if (!e) e = cudaEventSynchronize(b);
    if (!e) e = cudaEventElapsedTime(&ms, a, b);
    if (!e && kernel_gbs) *kernel_gbs = (double)bytes * iters / (ms * 1e-3) / 1e9;
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (e) return cuda_fail(h, e, "host link probe");
    return PE_OK;
}

pe_status pe_profile_enable(pe_handle* h, int32_t on) {
    if (!h) return PE_ERR_INVALID;
    if (on) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e) return cuda_fail(h, e, "synchronize");
        h->marks.clear();
        h->pool_used = 0;
        for (int i = 0; i < P_NUM; ++i) {
            h->prof_ms[i] = 0;
            h->prof_n[i] = 0;
        }
    }
    h->prof_on = on != 0;
    return PE_OK;
}

pe_status pe_profile_read(pe_handle* h, pe_profile_t* out) {
    if (!h || !out) return PE_ERR_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    if (e) return cuda_fail(h, e, "synchronize");
    drain_marks(h);
    std::memset(out, 0, sizeof(*out));
    for (int i = 0; i < P_NUM && i < PE_PROF_KINDS; ++i) {
        out->name[i] = kProfNames[i];
        out->launches[i] = h->prof_n[i];
        out->total_ms[i] = h->prof_ms[i];
    }
    return PE_OK;
}

void pe_destroy(pe_handle* h) {
    if (!h) return;
    cudaDeviceSynchronize();
    for (auto ev : h->pool) cudaEventDestroy(ev);
    if (h->owns_store && h->store_host) cudaFreeHost(h->store_host);
    if (h->external_store && h->store_host) unregister_external(h->store_host);
    delete h;
}

const char* pe_last_error(pe_handle* h) { return h ? h->last_error.c_str() : g_create_error.c_str(); }

}  // extern "C"
