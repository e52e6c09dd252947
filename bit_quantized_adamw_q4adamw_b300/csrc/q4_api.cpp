// C ABI of the q4adamw library: validation, host scalars, workspace layout,
// descriptor upload and kernel launches.  See include/q4adamw.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "q4_internal.h"

namespace {

using q4::DevTensor;

thread_local int g_last_cuda = 0;
thread_local long long g_wait_cycles = q4::kDefaultWaitCycles;   // q4adamw_set_stage_wait_limit

int cuda_fail(cudaError_t e) {
    g_last_cuda = (int)e;
    return Q4_ECUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t nblocks(int64_t numel) { return (numel + q4::kBlock - 1) / q4::kBlock; }

bool is_factored(const q4adamw_tensor_t& t, int recipe) {
    return recipe == Q4_RECIPE_FACTORED && (t.flags & Q4_T_FACTORED);
}

int check_recipe(int recipe) {
    return (recipe == Q4_RECIPE_ZIP_SR || recipe == Q4_RECIPE_ZE_EDEN || recipe == Q4_RECIPE_FACTORED ||
            recipe == Q4_RECIPE_TORCHAO)
               ? Q4_OK
               : Q4_ERECIPE;
}

// Codebook ids of a recipe's moments (listing page Table 2).
int m_book(int recipe) { return recipe == Q4_RECIPE_TORCHAO ? 3 : 0; }
int v_book(int recipe) {
    return recipe == Q4_RECIPE_ZIP_SR ? 1 : recipe == Q4_RECIPE_TORCHAO ? 4 : 2;
}

// Shape-only checks (host-only entry points).  A data-parallel shard of a
// factored parameter (dp) need not hold whole rows: check_dp checks its
// parameter's shape instead.
int check_shape(const q4adamw_tensor_t& t, int recipe, bool dp = false) {
    if (t.numel < 0) return Q4_ESHAPE;
    if (t.elem_offset % q4::kBlock) return Q4_ESHAPE;
    if (is_factored(t, recipe) && !dp) {
        if (t.rows < 1 || (t.numel > 0 && t.numel % t.rows)) return Q4_ESHAPE;
    }
    return Q4_OK;
}

// Full pointer checks for calls that touch device memory.
int check_tensor(const q4adamw_tensor_t& t, int recipe, bool need_grad, bool dp = false) {
    int rc = check_shape(t, recipe, dp);
    if (rc) return rc;
    if (t.numel == 0) return Q4_OK;
    if (!t.param || !t.m_codes || !t.m_scale) return Q4_EINVAL;
    if (need_grad && !t.grad) return Q4_EINVAL;
    if (!aligned(t.param, 16) || !aligned(t.m_codes, 16) || !aligned(t.m_scale, 4)) return Q4_EALIGN;
    if (t.grad && !aligned(t.grad, 16)) return Q4_EALIGN;
    if (t.param_bf16 && !aligned(t.param_bf16, 16)) return Q4_EALIGN;
    if (is_factored(t, recipe)) {
        if (!t.v_row || !t.v_col) return Q4_EINVAL;
        if (!aligned(t.v_row, 4) || !aligned(t.v_col, 4)) return Q4_EALIGN;
    } else {
        if (!t.v_codes || !t.v_scale) return Q4_EINVAL;
        if (!aligned(t.v_codes, 16) || !aligned(t.v_scale, 4)) return Q4_EALIGN;
    }
    return Q4_OK;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int64_t n_slabs(int64_t rows) { return (rows + q4::kSlabRows - 1) / q4::kSlabRows; }
int64_t n_segs(int64_t cols) { return (cols + q4::kSegCols - 1) / q4::kSegCols; }

// Where a factored tensor's elements sit in its parameter's [rows, cols]
// matrix.  A whole tensor (full_numel NULL) is the matrix [rows, numel/rows]
// from element 0; a data-parallel shard holds the elements [elem_offset,
// elem_offset + numel) of the matrix [rows, full_numel[i] / rows].  `fact`:
// the tensor keeps factored statistics in this call (a shard does even when
// it holds no element, as every rank updates the replicated R and C).
struct Geo {
    bool fact = false;
    int64_t rows = 0, cols = 0, fbase = 0;
    int64_t tiles = 0, partials = 0;   // statistics-pass tiles and partial-sum floats
};

Geo geometry(const q4adamw_tensor_t& t, int recipe, const int64_t* full_numel, int i) {
    Geo g;
    const int64_t full = full_numel ? full_numel[i] : t.numel;
    if (!is_factored(t, recipe) || full <= 0 || t.rows < 1) return g;
    g.fact = true;
    g.rows = t.rows;
    g.cols = full / t.rows;
    g.fbase = full_numel ? (int64_t)t.elem_offset : 0;
    int64_t r_first = 0, cov = 0;
    if (t.numel > 0) q4::covered_rows(g.fbase, t.numel, g.cols, &r_first, &cov);
    g.tiles = n_slabs(cov) * n_segs(g.cols);
    g.partials = n_slabs(cov) * g.cols + cov * n_segs(g.cols);
    return g;
}

// Data-parallel calls: the shape checks of a shard of a factored parameter
// (its matrix [rows, full_numel[i] / rows] holds the shard's elements
// [elem_offset, elem_offset + numel)), and R and C present even in a shard
// that holds no element.
int check_dp(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel) {
    if (!full_numel) return Q4_OK;
    for (int i = 0; i < n; ++i) {
        if (!is_factored(t[i], recipe)) continue;
        const int64_t full = full_numel[i];
        if (full < 0 || t[i].rows < 1 || (full > 0 && full % t[i].rows)) return Q4_ESHAPE;
        if ((int64_t)t[i].elem_offset > full || t[i].numel > full - (int64_t)t[i].elem_offset) return Q4_ESHAPE;
        if (full > 0) {
            if (!t[i].v_row || !t[i].v_col) return Q4_EINVAL;
            if (!aligned(t[i].v_row, 4) || !aligned(t[i].v_col, 4)) return Q4_EALIGN;
        }
    }
    return Q4_OK;
}

// Workspace layout, all offsets 256-B aligned.  The uploaded part is rewritten
// from a zeroed host image every step, which also clears the status word.
struct Layout {
    int64_t status, desc, pairs, rows, tiles, cols, fids;  // uploaded part
    int64_t desc2, pairs2;   // factored recipe: descriptors factored-first, and the two subsets' prefixes
    int64_t upload_bytes;
    int64_t rbar, colpart;                         // device-only part
    int64_t total;
    int n_factored;
    int64_t colpart_floats;
};

Layout make_layout(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel = nullptr) {
    Layout L{};
    int64_t off = 0;
    L.status = off; off = round_up(off + 4, 256);
    L.desc = off;  off = round_up(off + (int64_t)n * (int64_t)sizeof(DevTensor), 256);
    L.pairs = off; off = round_up(off + (int64_t)(n + 1) * 8, 256);
    L.rows = off;  off = round_up(off + (int64_t)(n + 1) * 8, 256);
    L.tiles = off; off = round_up(off + (int64_t)(n + 1) * 8, 256);
    L.cols = off;  off = round_up(off + (int64_t)(n + 1) * 8, 256);
    L.fids = off;  off = round_up(off + (int64_t)(n > 0 ? n : 1) * 4, 256);
    L.desc2 = off; off = round_up(off + (int64_t)n * (int64_t)sizeof(DevTensor), 256);
    L.pairs2 = off; off = round_up(off + (int64_t)(n + 2) * 8, 256);
    L.upload_bytes = off;
    L.rbar = off;  off = round_up(off + (int64_t)(n > 0 ? n : 1) * 16, 256);   // {mean(R), 1/mean(R), fast, 0}
    L.colpart = off;
    int64_t cp = 0;
    for (int i = 0; i < n; ++i) {
        const Geo g = geometry(t[i], recipe, full_numel, i);
        if (g.fact) {
            L.n_factored++;
            cp += g.partials;
        }
    }
    L.colpart_floats = cp;
    off = round_up(off + cp * 4, 256);
    L.total = off;
    return L;
}

// Workspace layout of q4adamw_grad_sqnorm (same status word at offset 0).
struct NormLayout {
    int64_t status, desc, prefix;                  // uploaded part
    int64_t upload_bytes;
    int64_t partials, tsums;                       // device-only part
    int64_t total;
    int64_t chunks;
};

int64_t norm_chunks(int64_t numel) {
    const int64_t tiles = (numel + 255) / 256;
    return (tiles + q4::kNormChunkTiles - 1) / q4::kNormChunkTiles;
}

NormLayout make_norm_layout(const q4adamw_tensor_t* t, int n) {
    NormLayout L{};
    int64_t off = 0;
    L.status = off; off = round_up(off + 4, 256);
    L.desc = off;   off = round_up(off + (int64_t)(n > 0 ? n : 1) * (int64_t)sizeof(q4::NormTensor), 256);
    L.prefix = off; off = round_up(off + (int64_t)(n + 1) * 8, 256);
    L.upload_bytes = off;
    for (int i = 0; i < n; ++i) L.chunks += norm_chunks(t[i].numel);
    L.partials = off; off = round_up(off + (L.chunks > 0 ? L.chunks : 1) * 4, 256);
    L.tsums = off;    off = round_up(off + (int64_t)(n > 0 ? n : 1) * 4, 256);
    L.total = off;
    return L;
}

// Host scalars of step t, each computed in double and rounded once to FP32.
struct Scalars {
    float c2, step_size, decay, omb1, omb2;
};
Scalars host_scalars(float lr, float beta1, float beta2, float wd, int64_t step) {
    const double dlr = lr, d1 = beta1, d2 = beta2, dwd = wd;
    const double bc1 = 1.0 - std::pow(d1, (double)step);
    const double bc2 = 1.0 - std::pow(d2, (double)step);
    Scalars s;
    s.c2 = (float)(1.0 / std::sqrt(bc2));
    s.step_size = (float)(dlr / bc1);
    s.decay = (float)(1.0 - dlr * dwd);
    s.omb1 = (float)(1.0 - d1);
    s.omb2 = (float)(1.0 - d2);
    return s;
}

q4::Tables* g_tabs[4] = {nullptr, nullptr, nullptr, nullptr};
std::once_flag g_tabs_once;

void build_all_tables() {
    for (int r = 0; r < 4; ++r) {
        q4::Tables* t = new (std::nothrow) q4::Tables;
        if (t && q4::build_tables(m_book(r), v_book(r), t)) g_tabs[r] = t;
        else delete t;
    }
}

// One immutable table set per recipe, built once.
q4::Tables* tables_for(int recipe) {
    std::call_once(g_tabs_once, build_all_tables);
    return g_tabs[recipe];
}

DevTensor make_dev(const q4adamw_tensor_t& t, int recipe, uint32_t call_flags, const Geo& g) {
    DevTensor d{};
    d.param = t.param;
    d.grad = t.grad;
    d.bf16 = t.param_bf16;
    d.mc = t.m_codes;
    d.ms = t.m_scale;
    d.vc = t.v_codes;
    d.vs = t.v_scale;
    d.vrow = t.v_row;
    d.vcol = t.v_col;
    d.numel = t.numel;
    d.rows = t.rows < 1 ? 1 : t.rows;
    d.cols = (t.numel > 0) ? t.numel / d.rows : 0;
    d.elem_offset = t.elem_offset;
    d.tensor_id = t.tensor_id;
    d.flags = 0;
    // listing page Table 2: LM-head SR in the final phase, except in the TorchAO
    // baseline; the Q4_M_SR_ALL variant rounds every first moment stochastically
    if (((t.flags & Q4_T_LM_HEAD) && (call_flags & Q4_LM_HEAD_SR_ACTIVE) && recipe != Q4_RECIPE_TORCHAO) ||
        (call_flags & Q4_M_SR_ALL))
        d.flags |= q4::DF_M_SR;
    if (is_factored(t, recipe)) {
        d.flags |= q4::DF_FACTORED;
        if (g.fact) {
            d.cols = g.cols;
            d.fbase = g.fbase;   // in place of the (absent) packed-v scales
        }
        // vector column loads and incremental (row, column) tracking in the step
        // kernel: columns a multiple of 8 (16-B aligned float4 runs) and at
        // least one tile (256) wide, rows within 32 bits
        if (d.cols % 8 == 0 && d.cols >= 256 && d.rows <= 0xFFFFFFFFll && aligned(t.v_col, 16))
            d.flags |= q4::DF_CVEC;
    }
    if (t.param_bf16) d.flags |= q4::DF_BF16;
    return d;
}

}  // namespace

namespace q4 {
int record_cuda_error(int cuda_error) { return cuda_fail((cudaError_t)cuda_error); }
}  // namespace q4

extern "C" {

int q4adamw_version(void) { return Q4ADAMW_STATE_FORMAT; }

const char* q4adamw_strerror(int status) {
    switch (status) {
        case Q4_OK: return "ok";
        case Q4_EINVAL: return "invalid argument";
        case Q4_EALIGN: return "misaligned pointer";
        case Q4_ESHAPE: return "invalid tensor shape";
        case Q4_ERECIPE: return "unknown recipe or codebook";
        case Q4_EVERSION: return "state header does not match this optimizer state format or recipe";
        case Q4_ECUDA: return "CUDA runtime error";
        case Q4_EWORKSPACE: return "workspace missing, too small or misaligned";
        default: return "unknown status";
    }
}

int q4adamw_last_cuda_error(void) { return g_last_cuda; }

int q4adamw_state_bytes(const q4adamw_tensor_t* t, int n, int recipe, int64_t* quantized, int64_t* scale_meta,
                        int64_t* total) {
    if (n < 0 || (n > 0 && !t)) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    int64_t q = 0, s = 0;
    for (int i = 0; i < n; ++i) {
        if (int rc = check_shape(t[i], recipe)) return rc;
        const int64_t nb = nblocks(t[i].numel);
        q += nb * 64;  // m codes
        s += nb * 4;   // m scales
        if (is_factored(t[i], recipe)) {
            if (t[i].numel > 0) s += (t[i].rows + t[i].numel / t[i].rows) * 4;
        } else {
            q += nb * 64;
            s += nb * 4;
        }
    }
    if (quantized) *quantized = q;
    if (scale_meta) *scale_meta = s;
    if (total) *total = q + s;
    return Q4_OK;
}

int q4adamw_workspace_bytes(const q4adamw_tensor_t* t, int n, int recipe, int64_t* bytes) {
    if (n < 0 || (n > 0 && !t) || !bytes) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    for (int i = 0; i < n; ++i)
        if (int rc = check_shape(t[i], recipe)) return rc;
    const int64_t a = make_layout(t, n, recipe).total, b = make_norm_layout(t, n).total;
    *bytes = a > b ? a : b;
    return Q4_OK;
}

int q4adamw_header_check(const q4adamw_header_t* h, int recipe) {
    if (!h) return Q4_EINVAL;
    if (h->magic != Q4ADAMW_MAGIC || h->format != Q4ADAMW_STATE_FORMAT || h->block != Q4ADAMW_BLOCK ||
        h->recipe != (uint32_t)recipe)
        return Q4_EVERSION;
    return Q4_OK;
}

}  // extern "C"

namespace {

// q4adamw_state_init and q4adamw_dp_state_init (full_numel: the shard
// geometry, NULL for whole tensors).
int state_init_impl(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                    q4adamw_header_t* header_out, void* stream) {
    if (n < 0 || (n > 0 && !t)) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    for (int i = 0; i < n; ++i)
        if (int rc = check_tensor(t[i], recipe, false, full_numel != nullptr)) return rc;
    if (int rc = check_dp(t, n, recipe, full_numel)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        const q4adamw_tensor_t& x = t[i];
        total += x.numel;
        const Geo g = geometry(x, recipe, full_numel, i);
        cudaError_t e = cudaSuccess;
        if (g.fact) {   // R and C of the whole parameter (an empty shard's too)
            e = cudaMemsetAsync(x.v_row, 0, (size_t)(g.rows * 4), s);
            if (e == cudaSuccess) e = cudaMemsetAsync(x.v_col, 0, (size_t)(g.cols * 4), s);
        }
        if (e == cudaSuccess && x.numel > 0) {
            const int64_t nb = nblocks(x.numel);
            e = cudaMemsetAsync(x.m_codes, 0, (size_t)(nb * 64), s);
            if (e == cudaSuccess) e = cudaMemsetAsync(x.m_scale, 0, (size_t)(nb * 4), s);
            if (e == cudaSuccess && !is_factored(x, recipe)) {
                e = cudaMemsetAsync(x.v_codes, 0, (size_t)(nb * 64), s);
                if (e == cudaSuccess) e = cudaMemsetAsync(x.v_scale, 0, (size_t)(nb * 4), s);
            }
        }
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (header_out) {
        header_out->magic = Q4ADAMW_MAGIC;
        header_out->format = Q4ADAMW_STATE_FORMAT;
        header_out->recipe = (uint32_t)recipe;
        header_out->block = Q4ADAMW_BLOCK;
        header_out->n_tensors = n;
        header_out->numel_total = total;
    }
    return Q4_OK;
}

}  // namespace

extern "C" {

int q4adamw_state_init(const q4adamw_tensor_t* t, int n, int recipe, q4adamw_header_t* header_out, void* stream) {
    return state_init_impl(t, n, recipe, nullptr, header_out, stream);
}

int q4adamw_dp_state_init(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                          q4adamw_header_t* header_out, void* stream) {
    return state_init_impl(t, n, recipe, full_numel, header_out, stream);
}

}  // extern "C"

namespace {

// Host image of the uploaded part of the workspace: descriptors, tile prefix
// sums, factored row/tile/column prefixes and ids, and the grouped copy for
// the two-launch split.  Returns the number of factored tensors.
struct Image {
    int nf = 0;
    int n_first = 0;           // tensors of the first group of the split (0: no split)
    uint32_t split_bit = 0;
};

Image build_image(const q4adamw_tensor_t* t, int n, int recipe, uint32_t flags, const int64_t* full_numel,
                  const Layout& L, std::vector<unsigned char>& img, char* ws) {
    Image im;
    img.assign((size_t)L.upload_bytes, 0);
    DevTensor* desc = reinterpret_cast<DevTensor*>(img.data() + L.desc);
    int64_t* pairs = reinterpret_cast<int64_t*>(img.data() + L.pairs);
    int64_t* rows = reinterpret_cast<int64_t*>(img.data() + L.rows);
    int64_t* tiles = reinterpret_cast<int64_t*>(img.data() + L.tiles);
    int64_t* cols = reinterpret_cast<int64_t*>(img.data() + L.cols);
    int32_t* fids = reinterpret_cast<int32_t*>(img.data() + L.fids);
    int64_t colpart_off = L.colpart;
    pairs[0] = rows[0] = tiles[0] = cols[0] = 0;
    for (int i = 0; i < n; ++i) {
        const Geo g = geometry(t[i], recipe, full_numel, i);
        desc[i] = make_dev(t[i], recipe, flags, g);
        const int64_t nb = nblocks(t[i].numel);
        pairs[i + 1] = pairs[i] + (nb + 1) / 2;
        rows[i + 1] = rows[i] + (g.fact ? g.rows : 0);
        cols[i + 1] = cols[i] + (g.fact ? g.cols : 0);
        tiles[i + 1] = tiles[i] + (g.fact ? g.tiles : 0);
        if (g.fact) {
            desc[i].rbar = reinterpret_cast<float*>(ws + L.rbar) + 4 * im.nf;
            desc[i].colpart = reinterpret_cast<float*>(ws + colpart_off);
            colpart_off += g.partials * 4;
            fids[im.nf++] = i;
        }
    }
    // Two launches where one instantiation does not suit every tensor: under
    // the factored recipe the factored tensors run on an instantiation without
    // the packed-v code and the 1-D ones on the general factored one; under
    // ZIP-SR / ZE-EDEN the tensors whose first moment is rounded
    // stochastically (the LM head during its SR phase) run on the m-SR
    // instantiation and the rest on the plain one.  desc2 holds the
    // descriptors of the first group first; pairs2 the two groups' prefix sums.
    im.split_bit = recipe == Q4_RECIPE_FACTORED ? (uint32_t)q4::DF_FACTORED
                   : (recipe == Q4_RECIPE_ZIP_SR || recipe == Q4_RECIPE_ZE_EDEN) ? (uint32_t)q4::DF_M_SR
                                                                                : 0u;
    if (im.split_bit) {
        DevTensor* desc2 = reinterpret_cast<DevTensor*>(img.data() + L.desc2);
        int64_t* pa = reinterpret_cast<int64_t*>(img.data() + L.pairs2);
        for (int i = 0; i < n; ++i)
            if (desc[i].flags & im.split_bit) desc2[im.n_first++] = desc[i];
        int k = im.n_first;
        for (int i = 0; i < n; ++i)
            if (!(desc[i].flags & im.split_bit)) desc2[k++] = desc[i];
        pa[0] = 0;
        for (int i = 0; i < im.n_first; ++i) pa[i + 1] = pa[i] + (nblocks(desc2[i].numel) + 1) / 2;
        int64_t* pb = pa + im.n_first + 1;
        pb[0] = 0;
        for (int i = im.n_first; i < n; ++i)
            pb[i - im.n_first + 1] = pb[i - im.n_first] + (nblocks(desc2[i].numel) + 1) / 2;
    }
    return im;
}

q4::FactoredParams factored_params(const Layout& L, const std::vector<unsigned char>& img, char* ws, int n, int nf,
                                   float beta2, float omb2, const float* sqnorm, float max_norm) {
    const int64_t* rows = reinterpret_cast<const int64_t*>(img.data() + L.rows);
    const int64_t* tiles = reinterpret_cast<const int64_t*>(img.data() + L.tiles);
    const int64_t* cols = reinterpret_cast<const int64_t*>(img.data() + L.cols);
    q4::FactoredParams fp{};
    fp.tensors = reinterpret_cast<const DevTensor*>(ws + L.desc);
    fp.row_prefix = reinterpret_cast<const int64_t*>(ws + L.rows);
    fp.tile_prefix = reinterpret_cast<const int64_t*>(ws + L.tiles);
    fp.col_prefix = reinterpret_cast<const int64_t*>(ws + L.cols);
    fp.factored_ids = reinterpret_cast<const int32_t*>(ws + L.fids);
    fp.n_tensors = n;
    fp.n_factored = nf;
    fp.total_rows = rows[n];
    fp.total_tiles = tiles[n];
    fp.total_cols = cols[n];
    fp.beta2 = beta2;
    fp.omb2 = omb2;
    fp.sqnorm = sqnorm;
    fp.max_norm = max_norm;
    return fp;
}

// q4adamw_step, q4adamw_step_clip and q4adamw_dp_step: sqnorm NULL means no
// clipping; full_numel: the data-parallel shard geometry (NULL: whole
// tensors); from_sums: the factored statistics come from `sums`, the sums
// over all shards, instead of this call's own gradients.
int step_impl(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps, float weight_decay,
              int64_t step, uint64_t seed, int recipe, uint32_t flags, const float* sqnorm, float max_norm,
              const int64_t* full_numel, bool from_sums, const float* sums, void* workspace, int64_t workspace_bytes,
              void* stream) {
    if (n < 0 || (n > 0 && !t)) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    if (step < 1 || step > 0xFFFFFFFFll) return Q4_EINVAL;
    if (flags & ~(Q4_LM_HEAD_SR_ACTIVE | Q4_M_SR_ALL | Q4_V_UPDATE_RTN | Q4_V_NEXT_R)) return Q4_EINVAL;
    if ((flags & (Q4_V_UPDATE_RTN | Q4_V_NEXT_R)) && recipe != Q4_RECIPE_ZIP_SR) return Q4_EINVAL;
    if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f)) return Q4_EINVAL;
    if (!(eps > 0.f) || !std::isfinite(eps) || !std::isfinite(lr) || !std::isfinite(weight_decay)) return Q4_EINVAL;
    for (int i = 0; i < n; ++i)
        if (int rc = check_tensor(t[i], recipe, true, full_numel != nullptr)) return rc;
    if (int rc = check_dp(t, n, recipe, full_numel)) return rc;
    const Layout L = make_layout(t, n, recipe, full_numel);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return Q4_EWORKSPACE;
    if (from_sums && L.n_factored > 0) {
        if (!sums) return Q4_EINVAL;
        if (!aligned(sums, 4)) return Q4_EALIGN;
    }
    q4::Tables* tabs = tables_for(recipe);
    if (!tabs) return Q4_EINVAL;
    if (n == 0) return Q4_OK;

    thread_local std::vector<unsigned char> img;
    char* ws = static_cast<char*>(workspace);
    const Image im = build_image(t, n, recipe, flags, full_numel, L, img, ws);
    const DevTensor* desc = reinterpret_cast<const DevTensor*>(img.data() + L.desc);
    const int64_t* pairs = reinterpret_cast<const int64_t*>(img.data() + L.pairs);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(workspace, img.data(), (size_t)L.upload_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);

    const Scalars hs = host_scalars(lr, beta1, beta2, weight_decay, step);
    const DevTensor* d_desc = reinterpret_cast<const DevTensor*>(ws + L.desc);

    if (im.nf > 0) {
        q4::FactoredParams fp = factored_params(L, img, ws, n, im.nf, beta2, hs.omb2, sqnorm, max_norm);
        int ce;
        if (from_sums) {
            fp.sums = const_cast<float*>(sums);
            ce = q4::launch_factored_from_sums(fp, stream);
        } else {
            ce = q4::launch_factored(fp, stream);
        }
        if (ce) return cuda_fail((cudaError_t)ce);
    }

    q4::StepParams p{};
    p.tensors = d_desc;
    p.status = reinterpret_cast<uint32_t*>(ws + L.status);
    p.pair_prefix = reinterpret_cast<const int64_t*>(ws + L.pairs);
    p.total_pairs = pairs[n];
    p.n_tensors = n;
    p.recipe = recipe;
    p.beta1 = beta1;
    p.beta2 = beta2;
    p.omb1 = hs.omb1;
    p.omb2 = hs.omb2;
    p.c2 = hs.c2;
    p.eps = eps;
    p.decay = hs.decay;
    p.step_size = hs.step_size;
    p.step = (uint32_t)step;
    // The fast square root / reciprocal need d = sqrt(v') c2 + eps inside
    // [2^-126, 2^126); with v' <= FLT_MAX and c2 <= 2^12 (beta2 < 1 in FP32)
    // that holds whenever eps lies in [2^-100, 2^60].
    p.fast_math = (eps >= 0x1p-100f && eps <= 0x1p60f) ? 1 : 0;
    p.v_update_rtn = (flags & Q4_V_UPDATE_RTN) ? 1 : 0;
    p.v_next_r = (flags & Q4_V_NEXT_R) ? 1 : 0;
    p.c2_next = host_scalars(lr, beta1, beta2, weight_decay, step + 1).c2;
    p.has_m_sr = 0;
    p.sqnorm = sqnorm;
    p.max_norm = max_norm;
    p.wait_cycles = g_wait_cycles;
    for (int i = 0; i < n; ++i) p.has_m_sr |= (desc[i].flags & q4::DF_M_SR) ? 1 : 0;
    p.x2_beta1 = make_float2(p.beta1, p.beta1);
    p.x2_beta2 = make_float2(p.beta2, p.beta2);
    p.x2_omb1 = make_float2(p.omb1, p.omb1);
    p.x2_omb2 = make_float2(p.omb2, p.omb2);
    p.x2_c2 = make_float2(p.c2, p.c2);
    p.x2_eps = make_float2(p.eps, p.eps);
    p.x2_decay = make_float2(p.decay, p.decay);
    p.x2_neg_step = make_float2(-p.step_size, -p.step_size);   // negation is exact
    q4::philox_round_keys(seed, p.round_keys);
    p.tab = *tabs;
    if (p.total_pairs == 0) return Q4_OK;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    // one group empty: the single launch below (the factored recipe with only
    // factored tensors still takes the factored-only instantiation)
    const int n_first = im.n_first;
    const bool split = im.split_bit != 0u && n_first > 0 && n_first < n;
    if (recipe == Q4_RECIPE_FACTORED && n_first == n) p.recipe = q4::kRecipeFactoredOnly;
    if (split) {
        const DevTensor* d2 = reinterpret_cast<const DevTensor*>(ws + L.desc2);
        const int64_t* pa = reinterpret_cast<const int64_t*>(ws + L.pairs2);
        const int64_t* ha = reinterpret_cast<const int64_t*>(img.data() + L.pairs2);
        const int sub_n[2] = {n_first, n - n_first};
        const int64_t sub_pairs[2] = {ha[n_first], ha[n_first + 1 + (n - n_first)]};
        for (int k = 0; k < 2; ++k) {
            if (sub_pairs[k] == 0) continue;
            q4::StepParams ps = p;
            ps.tensors = d2 + (k == 0 ? 0 : n_first);
            ps.pair_prefix = pa + (k == 0 ? 0 : n_first + 1);
            ps.n_tensors = sub_n[k];
            ps.total_pairs = sub_pairs[k];
            if (recipe == Q4_RECIPE_FACTORED) ps.recipe = k == 0 ? q4::kRecipeFactoredOnly : Q4_RECIPE_FACTORED;
            else ps.has_m_sr = k == 0 ? 1 : 0;
            if (int ce = q4::launch_step(ps, q4::step_grid_size(dev, ps.total_pairs), stream))
                return cuda_fail((cudaError_t)ce);
        }
        return Q4_OK;
    }
    const int grid = q4::step_grid_size(dev, p.total_pairs);
    if (int ce = q4::launch_step(p, grid, stream)) return cuda_fail((cudaError_t)ce);
    return Q4_OK;
}

}  // namespace

extern "C" {

int q4adamw_step(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps, float weight_decay,
                 int64_t step, uint64_t seed, int recipe, uint32_t flags, void* workspace, int64_t workspace_bytes,
                 void* stream) {
    return step_impl(t, n, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags, nullptr, 1.f, nullptr,
                     false, nullptr, workspace, workspace_bytes, stream);
}

int q4adamw_step_clip(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps,
                      float weight_decay, int64_t step, uint64_t seed, int recipe, uint32_t flags,
                      float max_grad_norm, const float* sqnorm, void* workspace, int64_t workspace_bytes,
                      void* stream) {
    if (!sqnorm || !aligned(sqnorm, 4)) return sqnorm ? Q4_EALIGN : Q4_EINVAL;
    if (!(max_grad_norm > 0.f) || !std::isfinite(max_grad_norm)) return Q4_EINVAL;
    return step_impl(t, n, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags, sqnorm, max_grad_norm,
                     nullptr, false, nullptr, workspace, workspace_bytes, stream);
}

int q4adamw_dp_workspace_bytes(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                               int64_t* bytes) {
    if (n < 0 || (n > 0 && !t) || !bytes) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    for (int i = 0; i < n; ++i)
        if (int rc = check_shape(t[i], recipe, full_numel != nullptr)) return rc;
    if (int rc = check_dp(t, n, recipe, full_numel)) return rc;
    const int64_t a = make_layout(t, n, recipe, full_numel).total, b = make_norm_layout(t, n).total;
    *bytes = a > b ? a : b;
    return Q4_OK;
}

int q4adamw_dp_sums_floats(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                           int64_t* floats) {
    if (n < 0 || (n > 0 && !t) || !floats) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    for (int i = 0; i < n; ++i)
        if (int rc = check_shape(t[i], recipe, full_numel != nullptr)) return rc;
    if (int rc = check_dp(t, n, recipe, full_numel)) return rc;
    int64_t f = 0;
    for (int i = 0; i < n; ++i) {
        const Geo g = geometry(t[i], recipe, full_numel, i);
        if (g.fact) f += g.rows + g.cols;
    }
    *floats = f;
    return Q4_OK;
}

int q4adamw_dp_factored_sums(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                             float max_grad_norm, const float* sqnorm, float* sums, void* workspace,
                             int64_t workspace_bytes, void* stream) {
    if (n < 0 || (n > 0 && !t)) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    if (sqnorm && (!(max_grad_norm > 0.f) || !std::isfinite(max_grad_norm))) return Q4_EINVAL;
    if (sqnorm && !aligned(sqnorm, 4)) return Q4_EALIGN;
    for (int i = 0; i < n; ++i) {
        if (int rc = check_shape(t[i], recipe, full_numel != nullptr)) return rc;
        if (is_factored(t[i], recipe) && t[i].numel > 0) {
            if (!t[i].grad) return Q4_EINVAL;
            if (!aligned(t[i].grad, 16)) return Q4_EALIGN;
        }
    }
    if (int rc = check_dp(t, n, recipe, full_numel)) return rc;
    const Layout L = make_layout(t, n, recipe, full_numel);
    if (L.n_factored == 0 || n == 0) return Q4_OK;
    if (!sums) return Q4_EINVAL;
    if (!aligned(sums, 4)) return Q4_EALIGN;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return Q4_EWORKSPACE;
    thread_local std::vector<unsigned char> img;
    char* ws = static_cast<char*>(workspace);
    const Image im = build_image(t, n, recipe, 0u, full_numel, L, img, ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(workspace, img.data(), (size_t)L.upload_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    q4::FactoredParams fp = factored_params(L, img, ws, n, im.nf, 0.f, 0.f, sqnorm, sqnorm ? max_grad_norm : 1.f);
    fp.sums = sums;
    if (int ce = q4::launch_factored_sums(fp, stream)) return cuda_fail((cudaError_t)ce);
    return Q4_OK;
}

int q4adamw_dp_step(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps,
                    float weight_decay, int64_t step, uint64_t seed, int recipe, uint32_t flags,
                    const int64_t* full_numel, const float* sums, float max_grad_norm, const float* sqnorm,
                    void* workspace, int64_t workspace_bytes, void* stream) {
    if (sqnorm && (!(max_grad_norm > 0.f) || !std::isfinite(max_grad_norm))) return Q4_EINVAL;
    if (sqnorm && !aligned(sqnorm, 4)) return Q4_EALIGN;
    // full_numel NULL: every tensor whole (matrix offset 0); its statistics
    // still come from sums
    return step_impl(t, n, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags, sqnorm,
                     sqnorm ? max_grad_norm : 1.f, full_numel, true, sums, workspace, workspace_bytes, stream);
}

int q4adamw_draws(uint64_t seed, int64_t step, uint32_t tensor_id, uint64_t idx0, uint32_t purpose, int64_t n,
                  uint32_t* out, void* stream) {
    if (n < 0 || (n > 0 && !out) || step < 1 || step > 0xFFFFFFFFll || purpose > 15u) return Q4_EINVAL;
    if (out && !aligned(out, 4)) return Q4_EALIGN;
    if (n == 0) return Q4_OK;
    if (int ce = q4::launch_draws(seed, (uint32_t)step, tensor_id, idx0, purpose, n, out, stream))
        return cuda_fail((cudaError_t)ce);
    return Q4_OK;
}

int q4adamw_grad_sqnorm(const q4adamw_tensor_t* t, int n, float* sqnorm, void* workspace, int64_t workspace_bytes,
                        void* stream) {
    if (n < 0 || (n > 0 && !t) || !sqnorm) return Q4_EINVAL;
    if (!aligned(sqnorm, 4)) return Q4_EALIGN;
    for (int i = 0; i < n; ++i) {
        if (t[i].numel < 0) return Q4_ESHAPE;
        if (t[i].numel > 0 && !t[i].grad) return Q4_EINVAL;
        if (t[i].grad && !aligned(t[i].grad, 16)) return Q4_EALIGN;
    }
    const NormLayout L = make_norm_layout(t, n);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return Q4_EWORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    thread_local std::vector<unsigned char> img;
    img.assign((size_t)L.upload_bytes, 0);
    q4::NormTensor* desc = reinterpret_cast<q4::NormTensor*>(img.data() + L.desc);
    int64_t* prefix = reinterpret_cast<int64_t*>(img.data() + L.prefix);
    prefix[0] = 0;
    for (int i = 0; i < n; ++i) {
        desc[i].grad = t[i].grad;
        desc[i].numel = t[i].numel;
        prefix[i + 1] = prefix[i] + norm_chunks(t[i].numel);
    }
    cudaError_t e = cudaMemcpyAsync(workspace, img.data(), (size_t)L.upload_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    char* ws = static_cast<char*>(workspace);
    q4::NormParams p{};
    p.tensors = reinterpret_cast<const q4::NormTensor*>(ws + L.desc);
    p.chunk_prefix = reinterpret_cast<const int64_t*>(ws + L.prefix);
    p.n_tensors = n;
    p.total_chunks = L.chunks;
    p.partials = reinterpret_cast<float*>(ws + L.partials);
    p.tensor_sums = reinterpret_cast<float*>(ws + L.tsums);
    p.out = sqnorm;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    if (int ce = q4::launch_grad_sqnorm(p, dev, stream)) return cuda_fail((cudaError_t)ce);
    return Q4_OK;
}

int q4adamw_grad_nonfinite(const q4adamw_tensor_t* t, int n, uint64_t* count, void* workspace,
                           int64_t workspace_bytes, void* stream) {
    if (n < 0 || (n > 0 && !t) || !count) return Q4_EINVAL;
    if (!aligned(count, 8)) return Q4_EALIGN;
    for (int i = 0; i < n; ++i) {
        if (t[i].numel < 0) return Q4_ESHAPE;
        if (t[i].numel > 0 && !t[i].grad) return Q4_EINVAL;
        if (t[i].grad && !aligned(t[i].grad, 16)) return Q4_EALIGN;
    }
    // the upload (descriptors and run prefixes) fits the gradient-norm layout
    const NormLayout L = make_norm_layout(t, n);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return Q4_EWORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    thread_local std::vector<unsigned char> img;
    img.assign((size_t)L.upload_bytes, 0);
    q4::NormTensor* desc = reinterpret_cast<q4::NormTensor*>(img.data() + L.desc);
    int64_t* prefix = reinterpret_cast<int64_t*>(img.data() + L.prefix);
    prefix[0] = 0;
    for (int i = 0; i < n; ++i) {
        desc[i].grad = t[i].grad;
        desc[i].numel = t[i].numel;
        prefix[i + 1] = prefix[i] + (t[i].numel + 7) / 8;
    }
    cudaError_t e = cudaMemcpyAsync(workspace, img.data(), (size_t)L.upload_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    char* ws = static_cast<char*>(workspace);
    q4::NonfiniteParams p{};
    p.tensors = reinterpret_cast<const q4::NormTensor*>(ws + L.desc);
    p.run_prefix = reinterpret_cast<const int64_t*>(ws + L.prefix);
    p.n_tensors = n;
    p.total_runs = prefix[n];
    p.out = reinterpret_cast<unsigned long long*>(count);
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    if (int ce = q4::launch_nonfinite(p, dev, stream)) return cuda_fail((cudaError_t)ce);
    return Q4_OK;
}

int q4adamw_set_stage_wait_limit(int64_t cycles) {
    if (cycles < 0) return Q4_EINVAL;
    g_wait_cycles = cycles == 0 ? q4::kDefaultWaitCycles : (long long)cycles;
    return Q4_OK;
}

int q4adamw_step_status(const void* workspace, uint32_t* status, void* stream) {
    if (!workspace || !status) return Q4_EINVAL;
    if (!aligned(workspace, 256)) return Q4_EWORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    *status = v;
    return Q4_OK;
}

int q4adamw_dequant_state(const q4adamw_tensor_t* t, int recipe, float* m_out, float* v_out, void* stream) {
    if (!t) return Q4_EINVAL;
    if (int rc = check_recipe(recipe)) return rc;
    if (int rc = check_tensor(*t, recipe, false)) return rc;
    if (t->numel == 0 || (!m_out && !v_out)) return Q4_OK;
    const DevTensor d = make_dev(*t, recipe, 0, geometry(*t, recipe, nullptr, 0));
    const q4::Codebook& nf4 = q4::codebook(m_book(recipe));
    const q4::Codebook& vb = q4::codebook(v_book(recipe));
    if (int ce = q4::launch_dequant(d, recipe, nf4.levels, vb.levels, m_out, v_out, stream))
        return cuda_fail((cudaError_t)ce);
    return Q4_OK;
}

int q4adamw_codebook(int which, float* levels, float* thresholds) {
    if (which < 0 || which > 4) return Q4_ERECIPE;
    const q4::Codebook& c = q4::codebook(which);
    if (levels) std::memcpy(levels, c.levels, sizeof c.levels);
    if (thresholds) std::memcpy(thresholds, c.thresholds, sizeof c.thresholds);
    return Q4_OK;
}

}  // extern "C"
