// api.cu -- the C ABI of libmnb (include/mnb.h): validation, the per-call
// dispatcher and the kernel launches.
//
// Dispatch follows the auto mode of "[WebGPU] Fuse rank-32 quantized LoRA with
// MatMulNBits" (onnxruntime PR 33370, commit message adding MatMulNBitsLoRA):
// chosen on every invocation from X's per-matrix row dimension M, independent
// of the batch size, with forced overrides kept for comparisons.  Few rows go
// to the weight-streaming decode kernel, more rows to the tensor-core prefill
// kernel; the threshold is a handle property (default 16).
//
// A non-empty adapter adds the LoRA down kernel first (normal stream order)
// and launches the matmul kernel after it with programmatic stream
// serialization, so the matmul streams weights while T is produced and waits
// (griddepcontrol.wait) only before it reads T.  Nothing here allocates or
// synchronizes, so mnb_run can be captured in a CUDA graph.
#include <mutex>
#include <new>

#include "mnb_internal.h"

namespace mnb {
// The library's device status word (one per device context; kernels receive
// its address).  See mnb_sync_status.
__device__ unsigned int g_status = 0u;
}  // namespace mnb

struct mnb_handle_s {
    mnb_desc d;
    int last_route;
};

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_init_mu;
// Per device: the context the setup below was done in (0 = none yet), the
// SM count and the status word's device address in that context.  A device
// address and a kernel attribute belong to one context: when the current
// context of the device changes (the primary context was reset and created
// again, or the caller made another context current) the setup runs again.
unsigned long long g_setup_ctx[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
unsigned int* g_status_ptr[kMaxDevices] = {};

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_desc(const mnb_desc* d) {
    if (!d) return MNB_ERR_ARG;
    if (d->N < 0 || d->K < 0) return MNB_ERR_ARG;
    if (d->N > (int64_t)INT32_MAX || d->K > (int64_t)INT32_MAX / 2) return MNB_ERR_UNSUPPORTED;
    if (d->bits != 2 && d->bits != 4 && d->bits != 8) return MNB_ERR_UNSUPPORTED;
    if (d->block_size != 32) return MNB_ERR_UNSUPPORTED;
    if (d->K % (d->bits == 2 ? 64 : 32) != 0) return MNB_ERR_UNSUPPORTED;  // packed rows of whole 16-byte units
    if (d->max_rank != 0 && d->max_rank != 32) return MNB_ERR_UNSUPPORTED;
    if (d->mode < MNB_MODE_AUTO || d->mode > MNB_MODE_FORCE_GEMM) return MNB_ERR_ARG;
    if ((d->flags & ~MNB_FLAG_EARLY_WEIGHTS) != 0) return MNB_ERR_ARG;
    return MNB_OK;
}

// Per-device setup in the current context: SM count, kernel attributes and
// the status word's address.  Returns MNB_OK and the device's SM count, or
// MNB_ERR_NO_DEVICE / MNB_ERR_CUDA.
int device_setup(int* sm_count, unsigned int** status = nullptr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MNB_ERR_NO_DEVICE;
    }
    int major = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MNB_ERR_NO_DEVICE;
    }
    if (major != 10) return MNB_ERR_NO_DEVICE;  // built for sm_103a only
    unsigned long long ctx = 0;
    if (mnb::current_context_id(&ctx) != cudaSuccess) return MNB_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_init_mu);
    if (g_setup_ctx[dev] != ctx) {
        int sms = 0;
        void* st = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return MNB_ERR_NO_DEVICE;
        }
        if (mnb::gemv_prepare() != cudaSuccess || mnb::gemm_prepare() != cudaSuccess ||
            mnb::lora_down_prepare() != cudaSuccess || mnb::decode_prepare() != cudaSuccess ||
            mnb::decode_mt_prepare() != cudaSuccess ||
            cudaGetSymbolAddress(&st, mnb::g_status) != cudaSuccess) {
            cudaGetLastError();
            return MNB_ERR_CUDA;
        }
        g_status_ptr[dev] = static_cast<unsigned int*>(st);
        g_sm_count[dev] = sms;
        g_setup_ctx[dev] = ctx;
    }
    *sm_count = g_sm_count[dev];
    if (status) *status = g_status_ptr[dev];
    return MNB_OK;
}

int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Idle SMs beside a prefill grid from which the LoRA down projection runs there.
constexpr int kIdleDownCtas = 8;

// Single-token decode kernel: rows split evenly over one CTA per SM, the
// adapter (if any) in the same launch.
void plan_decode(const mnb_desc& d, int rank, int sms, mnb_plan_info* p) {
    int ctas, SR, ring;
    size_t smem;
    mnb::decode_geometry((int)d.N, (int)d.K, d.bits, rank > 0, sms, &ctas, &SR, &ring, &smem);
    p->route = MNB_ROUTE_GEMV;
    p->lora_kernel = 0;
    p->grid_x = ctas;
    p->grid_y = 1;
    p->block_threads = rank > 0 ? 320 : 288;
    p->rows_per_cta = (int)((d.N + ctas - 1) / ctas);
    p->k_splits = SR;
    p->tokens_per_cta = 1;
}

// Decode kernel for 2 .. 16 token rows: rows split evenly over one CTA per SM,
// the token rows as the MMA's N.
void plan_decode_mt(const mnb_desc& d, int64_t Mt, int sms, mnb_plan_info* p) {
    int ctas, parts, ring;
    size_t smem;
    mnb::decode_mt_geometry((int)d.N, (int)d.K, d.bits, (int)Mt, true, sms, &ctas, &parts, &ring, &smem);
    p->route = MNB_ROUTE_GEMV;
    p->lora_kernel = 0;
    p->grid_x = ctas;
    p->grid_y = 1;
    p->block_threads = 576;  // 16 consumer warps, the producer and the reducer
    p->rows_per_cta = (int)((d.N + ctas - 1) / ctas);
    p->k_splits = 16;
    p->tokens_per_cta = Mt <= 8 ? 8 : 16;
}

// Which decode kernel streams the weights of a decode-route call: the
// single-token kernel, the kernel for 2 .. 16 token rows, or (0) the general
// multi-token kernel.  fused_ok: FP16 activations; q8_adapter: an INT8 adapter
// (the single-token kernel takes it, the kernel for 2 .. 16 rows does not).
enum { kDecGeneral = 0, kDecSingle = 1, kDecMulti = 2 };
int decode_kind(const mnb_desc& d, int64_t Mt, int rank, int sms, bool fused_ok, bool q8_adapter = false) {
    if (!fused_ok) return kDecGeneral;
    if (mnb::decode_supported(d.bits, Mt, (int)d.K, d.N, rank > 0, sms)) return kDecSingle;
    if (rank > 0 && q8_adapter) return kDecGeneral;
    if (mnb::decode_mt_supported(d.bits, Mt, (int)d.K, rank > 0)) return kDecMulti;
    return kDecGeneral;
}

// Decode-kernel geometry: balanced row ranges, one CTA per SM and token group.
void plan_gemv(const mnb_desc& d, int64_t Mt, int sms, mnb_plan_info* p) {
    int ctas, R, CH, tok, threads;
    mnb::gemv_geometry((int)d.N, (int)d.K, d.bits, (int)Mt, sms, &ctas, &R, &CH, &tok, &threads);
    p->route = MNB_ROUTE_GEMV;
    p->grid_x = ctas;
    p->grid_y = cdiv(Mt, tok);
    p->block_threads = threads;
    p->rows_per_cta = R;
    p->k_splits = CH;
    p->tokens_per_cta = tok;
}

// Prefill-kernel geometry: 128 weight rows x up to 256 token rows per tile,
// one persistent CTA per SM.
void plan_gemm(const mnb_desc& d, int64_t Mt, int sms, mnb_plan_info* p) {
    const int tok = mnb::gemm_token_tile((int)Mt);
    const int ntiles = cdiv(d.N, 128) * cdiv(Mt, tok);
    const int split = mnb::gemm_split((int)d.N, (int)Mt, (int)d.K, sms);
    p->route = MNB_ROUTE_GEMM;
    if (split > 1)
        p->grid_x = ntiles * split;  // one cluster of `split` CTAs per tile
    else
        p->grid_x = ntiles < sms ? ntiles : (sms > 0 ? sms : 1);
    p->grid_y = 1;
    p->block_threads = mnb::gemm_threads();
    p->rows_per_cta = 128;
    p->k_splits = split;
    p->tokens_per_cta = tok;
}

// fused_ok: the call's variant can run on the single-token decode kernel (FP16 or
// no adapter, FP16 activations, one projection).
int make_plan(const mnb_desc& d, int64_t batch, int64_t M, int rank, int sms, mnb_plan_info* p,
              bool fused_ok = true, bool q8_adapter = false) {
    *p = mnb_plan_info{};
    const int64_t Mt = batch * M;
    if (Mt == 0 || d.N == 0) {
        p->route = MNB_ROUTE_NONE;
        return MNB_OK;
    }
    if (d.K == 0) {
        p->route = MNB_ROUTE_FILL;
        return MNB_OK;
    }
    const int thr = d.gemv_max_m > 0 ? d.gemv_max_m : 16;
    int route = M <= thr ? MNB_ROUTE_GEMV : MNB_ROUTE_GEMM;
    if (d.mode == MNB_MODE_FORCE_GEMV) route = MNB_ROUTE_GEMV;
    if (d.mode == MNB_MODE_FORCE_GEMM) route = MNB_ROUTE_GEMM;
    if (route == MNB_ROUTE_GEMV) {
        const int kind = decode_kind(d, Mt, rank, sms, fused_ok, q8_adapter);
        if (kind == kDecSingle) {
            plan_decode(d, rank, sms, p);
            return MNB_OK;
        }
        if (kind == kDecMulti) {
            plan_decode_mt(d, Mt, sms, p);
            p->lora_kernel = rank > 0 ? 1 : 0;
            return MNB_OK;
        }
    }
    if (route == MNB_ROUTE_GEMV)
        plan_gemv(d, Mt, sms, p);
    else
        plan_gemm(d, Mt, sms, p);
    p->lora_kernel = rank > 0 ? 1 : 0;
    return MNB_OK;
}

}  // namespace

extern "C" {

int mnb_create(const mnb_desc* desc, mnb_handle* out) {
    if (!out) return MNB_ERR_ARG;
    *out = nullptr;
    const int rc = validate_desc(desc);
    if (rc != MNB_OK) return rc;
    mnb_handle h = new (std::nothrow) mnb_handle_s;
    if (!h) return MNB_ERR_ARG;
    h->d = *desc;
    h->last_route = MNB_ROUTE_NONE;
    *out = h;
    return MNB_OK;
}

void mnb_destroy(mnb_handle h) { delete h; }

int mnb_last_route(mnb_handle h) { return h ? h->last_route : MNB_ROUTE_NONE; }

int mnb_plan(mnb_handle h, int64_t batch, int64_t M, int32_t rank, int32_t sm_count, mnb_plan_info* out) {
    if (!h || !out || batch < 0 || M < 0) return MNB_ERR_ARG;
    if (batch > 0 && M > INT32_MAX / batch) return MNB_ERR_UNSUPPORTED;
    if (rank != 0 && rank != 32) return MNB_ERR_UNSUPPORTED;
    if (rank > h->d.max_rank) return MNB_ERR_ARG;
    int sms = sm_count;
    if (sms <= 0) {  // the current device
        const int rc = device_setup(&sms);
        if (rc != MNB_OK) return rc;
    }
    return make_plan(h->d, batch, M, rank, sms, out);
}

}  // extern "C"

namespace {

// The adapter of one call: FP16 A [K, 32] and B [N, 32], or INT8 block-32
// weights Aq [32, K] / Bq [N, 32] with their scales and zero points.
struct Adapter {
    const void *A, *B;
    const void *Aq, *As, *Az, *Bq, *Bs, *Bz;
    bool q8;
};

// q8x: the int8-activation base (decode kernel for every M).  noalloc: T goes
// to the library's fixed scratch (mnb_run_noalloc); T_ws is then unused.
int run_impl(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const Adapter& ad,
             int32_t rank, const void* bias, void* Y, void* T_ws, int64_t batch, int64_t M, void* stream,
             bool q8x = false, bool noalloc = false) {
    if (!h || batch < 0 || M < 0) return MNB_ERR_ARG;
    const mnb_desc& d = h->d;
    if (batch > 0 && M > INT32_MAX / batch) return MNB_ERR_UNSUPPORTED;
    const int64_t Mt = batch * M;
    if (Mt > 0 && d.N > 0 && Mt * d.N > ((int64_t)1 << 40)) return MNB_ERR_UNSUPPORTED;
    // empty adapter: rank 0, or both adapter weights NULL
    if (rank != 0 && rank != 32) return MNB_ERR_UNSUPPORTED;
    const void* down = ad.q8 ? ad.Aq : ad.A;
    const void* up = ad.q8 ? ad.Bq : ad.B;
    if (down == nullptr && up == nullptr) rank = 0;
    if (rank > 0) {
        if (rank > d.max_rank) return MNB_ERR_ARG;
        if (!down || !up || (!T_ws && !noalloc)) return MNB_ERR_ARG;
        if (ad.q8 && (!ad.As || !ad.Bs)) return MNB_ERR_ARG;
    }
    if (Mt > 0 && d.N > 0) {
        if (!Y) return MNB_ERR_ARG;
        // Wq == NULL with K > 0: an empty packed weight (scales, zp unused)
        if (d.K > 0 && Wq && (!X || !scales)) return MNB_ERR_ARG;
        if (d.K > 0 && !Wq && rank > 0 && !X) return MNB_ERR_ARG;
    }
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(scales) || !aligned16(zp) || !aligned16(Y) ||
        !aligned16(bias) || (rank > 0 && (!aligned16(down) || !aligned16(up) || !aligned16(T_ws))) ||
        (rank > 0 && ad.q8 && (!aligned16(ad.As) || !aligned16(ad.Az) || !aligned16(ad.Bs) || !aligned16(ad.Bz))))
        return MNB_ERR_ALIGN;
    const __half* biash = static_cast<const __half*>(bias);
    const uint8_t* Bq8 = rank > 0 && ad.q8 ? static_cast<const uint8_t*>(ad.Bq) : nullptr;
    const __half* Bs8 = Bq8 ? static_cast<const __half*>(ad.Bs) : nullptr;
    const uint8_t* Bz8 = Bq8 ? static_cast<const uint8_t*>(ad.Bz) : nullptr;
    unsigned int* status = nullptr;  // the device's status word (set up below)
    auto launch_down = [&](const __half* Xh, __half* Th, bool early, cudaStream_t st, int max_ctas = 0) {
        return ad.q8 ? mnb::lora_down_q8_launch(Xh, static_cast<const uint8_t*>(ad.Aq),
                                                static_cast<const __half*>(ad.As),
                                                static_cast<const uint8_t*>(ad.Az), Th, (int)Mt, (int)d.K, early, st,
                                                max_ctas, status)
                     : mnb::lora_down_launch(Xh, static_cast<const __half*>(ad.A), Th, (int)Mt, (int)d.K, early, st,
                                             max_ctas, status);
    };

    mnb_plan_info p;
    int sms = 0;
    if (Mt > 0 && d.N > 0) {
        const int rc = device_setup(&sms, &status);
        if (rc != MNB_OK) return rc;
        if (noalloc && rank > 0) {
            if (Mt > mnb::kNoallocMaxRows) return MNB_ERR_UNSUPPORTED;  // beyond the fixed scratch
            __half* Tfix = nullptr;
            const int rs = mnb::noalloc_scratch(&Tfix);
            if (rs != MNB_OK) return rs;
            T_ws = Tfix;
        }
    }
    make_plan(d, batch, M, rank, sms, &p, !q8x, rank > 0 && ad.q8);
    if (q8x && (p.route == MNB_ROUTE_GEMV || p.route == MNB_ROUTE_GEMM)) {
        plan_gemv(d, Mt, sms, &p);  // integer dots on the decode kernel, 8-token tiles
        p.tokens_per_cta = 8;
        p.grid_y = cdiv(Mt, 8);
        p.lora_kernel = rank > 0 ? 1 : 0;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;

    if (p.route == MNB_ROUTE_NONE) {
        h->last_route = MNB_ROUTE_NONE;
        return MNB_OK;
    }
    if (p.route != MNB_ROUTE_FILL && !Wq) {
        // empty packed weight: zeros or the broadcast bias, plus the adapter term
        if (rank == 0) {
            p.route = MNB_ROUTE_FILL;
        } else {
            e = launch_down(static_cast<const __half*>(X), static_cast<__half*>(T_ws), false, st);
            if (e == cudaSuccess)
                e = mnb::lora_up_launch(static_cast<const __half*>(T_ws), static_cast<const __half*>(ad.B), Bq8, Bs8,
                                        Bz8, biash, static_cast<__half*>(Y), (int)Mt, (int)d.N, st);
            if (e != cudaSuccess) return MNB_ERR_CUDA;
            h->last_route = MNB_ROUTE_FILL;
            return MNB_OK;
        }
    }
    if (p.route == MNB_ROUTE_FILL) {
        e = biash ? mnb::fill_bias_launch(static_cast<__half*>(Y), biash, (size_t)Mt, (size_t)d.N, st)
                  : mnb::fill_zero_launch(static_cast<__half*>(Y), (size_t)Mt * (size_t)d.N, st);
        if (e == cudaSuccess && rank > 0) e = mnb::fill_zero_launch(static_cast<__half*>(T_ws), (size_t)Mt * 32, st);
        if (e != cudaSuccess) return MNB_ERR_CUDA;
        h->last_route = MNB_ROUTE_FILL;
        return MNB_OK;
    }

    const __half* Xh = static_cast<const __half*>(X);
    __half* Th = static_cast<__half*>(T_ws);
    // Programmatic dependent launch.  With early weights the first kernel of a
    // call may start before the work queued ahead of it has completed: it
    // streams weights at once and reads X only after griddepcontrol.wait.  The
    // LoRA down kernel lets the matmul kernel start only after its own wait,
    // so behind it the matmul kernel reads X at once and waits only for T.
    const bool early = (d.flags & MNB_FLAG_EARLY_WEIGHTS) != 0;
    const int kind = p.route == MNB_ROUTE_GEMV ? decode_kind(d, Mt, rank, sms, !q8x, rank > 0 && ad.q8) : kDecGeneral;
    if (kind != kDecGeneral) {
        // one launch: the single-token decode kernel (base and adapter), or the
        // decode kernel for 2 .. 16 token rows (behind the LoRA down kernel with an
        // adapter: X is then complete when it starts, only T is waited for)
        const bool down = kind == kDecMulti && rank > 0;
        if (down) {
            e = launch_down(Xh, Th, early, st);
            if (e != cudaSuccess) return MNB_ERR_CUDA;
        }
        mnb::DecodeArgs a = {};
        a.nseg = 1;
        a.NR = (int)d.N;
        a.seg[0] = mnb::DecSeg{0, (int)d.N, static_cast<const uint8_t*>(Wq), static_cast<const __half*>(scales),
                               static_cast<const uint8_t*>(zp), biash, static_cast<__half*>(Y)};
        a.X = Xh;
        a.A = rank > 0 && !ad.q8 ? static_cast<const __half*>(ad.A) : nullptr;
        a.B = rank > 0 && !ad.q8 ? static_cast<const __half*>(ad.B) : nullptr;
        if (rank > 0 && ad.q8) {  // INT8 adapter: single-token kernel only
            a.Aq = static_cast<const uint8_t*>(ad.Aq);
            a.As = static_cast<const __half*>(ad.As);
            a.Az = static_cast<const uint8_t*>(ad.Az);
            a.Bq = Bq8;
            a.Bs = Bs8;
            a.Bz = Bz8;
        }
        a.T = rank > 0 ? Th : nullptr;
        a.K = (int)d.K;
        a.bits = d.bits;
        a.Mt = (int)Mt;
        a.x_wait = early && !down ? 1 : 0;
        a.status = status;
        e = kind == kDecSingle ? mnb::decode_launch(a, rank, sms, early, st)
                               : mnb::decode_mt_launch(a, sms, early || down, st);
        if (e == cudaErrorNotSupported) return MNB_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return MNB_ERR_CUDA;
        h->last_route = p.route;
        return MNB_OK;
    }
    const bool lora_kernel = rank > 0;
    if (lora_kernel) {
        // A prefill grid well short of the SM count leaves SMs idle: the down
        // projection runs there, beside the prefill kernel (which needs T only for
        // its last stage), instead of first holding SMs that kernel waits for.
        const int idle = p.route == MNB_ROUTE_GEMM && p.k_splits <= 1 ? sms - p.grid_x : 0;
        e = launch_down(Xh, Th, early, st, idle >= kIdleDownCtas ? idle : 0);
        if (e != cudaSuccess) return MNB_ERR_CUDA;
    }
    const bool pdl = lora_kernel || early;
    if (p.route == MNB_ROUTE_GEMV) {
        mnb::GemvArgs a = {};
        a.nseg = 1;
        a.G = cdiv(d.N, 16);
        a.seg[0] = mnb::GemvSeg{0, (int)d.N, static_cast<const uint8_t*>(Wq), static_cast<const __half*>(scales),
                                static_cast<const uint8_t*>(zp), biash, static_cast<__half*>(Y)};
        a.X = Xh;
        a.T = Th;
        a.B = static_cast<const __half*>(ad.B);
        a.Bq = Bq8;
        a.Bs = Bs8;
        a.Bz = Bz8;
        a.Mt = (int)Mt;
        a.K = (int)d.K;
        a.R = p.rows_per_cta;
        a.CH = p.k_splits;
        a.rank = rank;
        // after the LoRA down kernel the preceding work is complete when this
        // kernel starts (see lora_down.cu): only T needs the wait
        a.x_wait = early && !lora_kernel ? 1 : 0;
        a.sms = sms;
        a.w3d = 0;
        a.status = status;
        e = q8x ? mnb::gemv_q8x_launch(a, p, d.bits, pdl, st) : mnb::gemv_launch(a, p, d.bits, pdl, st);
        if (e == cudaErrorNotSupported) return MNB_ERR_UNSUPPORTED;
    } else {
        mnb::GemmArgs a;
        a.X = Xh;
        a.Wq = static_cast<const uint8_t*>(Wq);
        a.S = static_cast<const __half*>(scales);
        a.Z = static_cast<const uint8_t*>(zp);
        a.T = Th;
        a.B = static_cast<const __half*>(ad.B);
        a.Bq = Bq8;
        a.Bs = Bs8;
        a.Bz = Bz8;
        a.bias = biash;
        a.Y = static_cast<__half*>(Y);
        a.Mt = (int)Mt;
        a.N = (int)d.N;
        a.K = (int)d.K;
        a.bits = d.bits;
        a.rank = rank;
        a.status = status;
        e = mnb::gemm_launch(a, p, pdl, early && !lora_kernel, st);
        if (e == cudaErrorNotSupported) return MNB_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return MNB_ERR_CUDA;
    h->last_route = p.route;
    return MNB_OK;
}

}  // namespace

namespace mnb {
int run_noalloc(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const void* A,
                const void* B, int32_t rank, void* Y, int64_t batch, int64_t M, void* stream) {
    return run_impl(h, X, Wq, scales, zp, Adapter{A, B, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, false},
                    rank, nullptr, Y, nullptr, batch, M, stream, false, true);
}
}  // namespace mnb

extern "C" {

int mnb_run(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const void* A,
            const void* B, int32_t rank, void* Y, void* T_ws, int64_t batch, int64_t M, void* stream) {
    return run_impl(h, X, Wq, scales, zp, Adapter{A, B, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, false},
                    rank, nullptr, Y, T_ws, batch, M, stream);
}

int mnb_run_bias(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const void* A,
                 const void* B, int32_t rank, const void* bias, void* Y, void* T_ws, int64_t batch, int64_t M,
                 void* stream) {
    return run_impl(h, X, Wq, scales, zp, Adapter{A, B, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, false},
                    rank, bias, Y, T_ws, batch, M, stream);
}

int mnb_run_qlora(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const void* Aq,
                  const void* A_scales, const void* A_zp, const void* Bq, const void* B_scales, const void* B_zp,
                  int32_t rank, const void* bias, void* Y, void* T_ws, int64_t batch, int64_t M, void* stream) {
    return run_impl(h, X, Wq, scales, zp, Adapter{nullptr, nullptr, Aq, A_scales, A_zp, Bq, B_scales, B_zp, true},
                    rank, bias, Y, T_ws, batch, M, stream);
}

int mnb_run_q8x(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const void* A,
                const void* B, int32_t rank, const void* bias, void* Y, void* T_ws, int64_t batch, int64_t M,
                void* stream) {
    return run_impl(h, X, Wq, scales, zp, Adapter{A, B, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, false},
                    rank, bias, Y, T_ws, batch, M, stream, true);
}

int mnb_check_wait_timeout(int64_t limit_cycles, void* stream) {
    if (limit_cycles < 1000 || limit_cycles > 4000000000LL) return MNB_ERR_ARG;
    int sms;
    unsigned int* status = nullptr;
    const int rc = device_setup(&sms, &status);
    if (rc != MNB_OK) return rc;
    return mnb::wait_check_launch(status, (long long)limit_cycles, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MNB_OK
               : MNB_ERR_CUDA;
}

int mnb_quantize_x(const void* X, int64_t Mt, int64_t K, void* Xq, void* Xs, void* stream) {
    if (Mt < 0 || K < 0) return MNB_ERR_ARG;
    if (K % 32 != 0) return MNB_ERR_UNSUPPORTED;
    if (Mt > INT32_MAX || K > INT32_MAX / 2) return MNB_ERR_UNSUPPORTED;
    if (Mt == 0 || K == 0) return MNB_OK;
    if (!X || !Xq || !Xs) return MNB_ERR_ARG;
    if (!aligned16(X) || !aligned16(Xq) || !aligned16(Xs)) return MNB_ERR_ALIGN;
    int sms;
    const int rc = device_setup(&sms);
    if (rc != MNB_OK) return rc;
    const cudaError_t e = mnb::quantize_x_launch(static_cast<const __half*>(X), (int)Mt, (int)K, static_cast<int8_t*>(Xq),
                                                 static_cast<float*>(Xs), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MNB_OK : MNB_ERR_CUDA;
}

int mnb_run_multi(mnb_handle h, const void* X, const mnb_projection* proj, int32_t nproj, int64_t batch, int64_t M,
                  void* stream) {
    if (!h || !proj || batch < 0 || M < 0) return MNB_ERR_ARG;
    if (nproj < 1 || nproj > mnb::kMaxSeg) return MNB_ERR_UNSUPPORTED;
    const mnb_desc& d = h->d;
    if (batch > 0 && M > INT32_MAX / batch) return MNB_ERR_UNSUPPORTED;
    const int64_t Mt = batch * M;
    int64_t total = 0;
    int nonempty = 0, with_zp = 0;
    for (int i = 0; i < nproj; ++i) {
        const mnb_projection& q = proj[i];
        if (q.N < 0 || q.N > (int64_t)INT32_MAX) return MNB_ERR_ARG;
        total += q.N;
        if (!aligned16(q.Wq) || !aligned16(q.scales) || !aligned16(q.zp) || !aligned16(q.bias) || !aligned16(q.Y))
            return MNB_ERR_ALIGN;
        if (Mt > 0 && q.N > 0) {
            if (!q.Y) return MNB_ERR_ARG;
            if (d.K > 0 && q.Wq) {
                if (!q.scales || !X) return MNB_ERR_ARG;
                ++nonempty;
                with_zp += q.zp ? 1 : 0;
            }
        }
    }
    if (total != d.N) return MNB_ERR_ARG;  // the handle describes the fused weight: N = sum of the projections
    if (with_zp != 0 && with_zp != nonempty) return MNB_ERR_UNSUPPORTED;  // zero points for all or none
    if (!aligned16(X)) return MNB_ERR_ALIGN;
    if (Mt > 0 && Mt * d.N > ((int64_t)1 << 40)) return MNB_ERR_UNSUPPORTED;
    if (Mt == 0 || d.N == 0) {
        h->last_route = MNB_ROUTE_NONE;
        return MNB_OK;
    }
    int sms = 0;
    unsigned int* status = nullptr;
    int rc = device_setup(&sms, &status);
    if (rc != MNB_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    // empty members (or K == 0): zeros or the broadcast bias, the shared fallback
    for (int i = 0; i < nproj && e == cudaSuccess; ++i) {
        const mnb_projection& q = proj[i];
        if (q.N == 0 || (d.K > 0 && q.Wq)) continue;
        __half* Yq = static_cast<__half*>(q.Y);
        e = q.bias ? mnb::fill_bias_launch(Yq, static_cast<const __half*>(q.bias), (size_t)Mt, (size_t)q.N, st)
                   : mnb::fill_zero_launch(Yq, (size_t)Mt * (size_t)q.N, st);
    }
    if (e != cudaSuccess) return MNB_ERR_CUDA;
    if (nonempty == 0) {
        h->last_route = MNB_ROUTE_FILL;
        return MNB_OK;
    }
    const bool early = (d.flags & MNB_FLAG_EARLY_WEIGHTS) != 0;
    mnb_plan_info p;
    make_plan(d, batch, M, 0, sms, &p);
    const int kind = p.route == MNB_ROUTE_GEMV ? decode_kind(d, Mt, 0, sms, true) : kDecGeneral;
    if (kind != kDecGeneral) {
        // up to 16 token rows: one decode launch over the nonempty members
        mnb::DecodeArgs a = {};
        int R = 0;
        for (int i = 0; i < nproj; ++i) {
            const mnb_projection& q = proj[i];
            if (q.N == 0 || !q.Wq) continue;
            a.seg[a.nseg++] = mnb::DecSeg{R, (int)q.N, static_cast<const uint8_t*>(q.Wq),
                                          static_cast<const __half*>(q.scales), static_cast<const uint8_t*>(q.zp),
                                          static_cast<const __half*>(q.bias), static_cast<__half*>(q.Y)};
            R += (int)q.N;
        }
        a.NR = R;
        a.X = static_cast<const __half*>(X);
        a.Mt = (int)Mt;
        a.K = (int)d.K;
        a.bits = d.bits;
        a.x_wait = early ? 1 : 0;
        a.status = status;
        e = kind == kDecSingle ? mnb::decode_launch(a, 0, sms, early, st) : mnb::decode_mt_launch(a, sms, early, st);
        if (e == cudaErrorNotSupported) return MNB_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return MNB_ERR_CUDA;
        h->last_route = p.route;
        return MNB_OK;
    }
    make_plan(d, batch, M, 0, sms, &p, false);
    if (p.route == MNB_ROUTE_GEMV) {
        // one launch over the nonempty members, each starting on a 16-row group
        mnb::GemvArgs a = {};
        int G = 0;
        for (int i = 0; i < nproj; ++i) {
            const mnb_projection& q = proj[i];
            if (q.N == 0 || !q.Wq) continue;
            a.seg[a.nseg++] = mnb::GemvSeg{G, (int)q.N, static_cast<const uint8_t*>(q.Wq),
                                           static_cast<const __half*>(q.scales), static_cast<const uint8_t*>(q.zp),
                                           static_cast<const __half*>(q.bias), static_cast<__half*>(q.Y)};
            G += cdiv(q.N, 16);
        }
        a.G = G;
        mnb_desc dv = d;
        dv.N = (int64_t)G * 16;  // the launch geometry of the members' row space
        make_plan(dv, batch, M, 0, sms, &p, false);
        a.X = static_cast<const __half*>(X);
        a.Mt = (int)Mt;
        a.K = (int)d.K;
        a.R = p.rows_per_cta;
        a.CH = p.k_splits;
        a.rank = 0;
        a.x_wait = early ? 1 : 0;
        a.sms = sms;
        a.status = status;
        e = mnb::gemv_launch(a, p, d.bits, early, st);
    } else {
        // prefill: one tensor-core launch per nonempty member (each long enough
        // that a launch costs nothing in comparison)
        for (int i = 0; i < nproj && e == cudaSuccess; ++i) {
            const mnb_projection& q = proj[i];
            if (q.N == 0 || !q.Wq) continue;
            mnb_desc dq = d;
            dq.N = q.N;
            mnb_plan_info pq;
            make_plan(dq, batch, M, 0, sms, &pq, false);
            mnb::GemmArgs a = {};
            a.X = static_cast<const __half*>(X);
            a.Wq = static_cast<const uint8_t*>(q.Wq);
            a.S = static_cast<const __half*>(q.scales);
            a.Z = static_cast<const uint8_t*>(q.zp);
            a.bias = static_cast<const __half*>(q.bias);
            a.Y = static_cast<__half*>(q.Y);
            a.Mt = (int)Mt;
            a.N = (int)q.N;
            a.K = (int)d.K;
            a.bits = d.bits;
            a.rank = 0;
            a.status = status;
            e = mnb::gemm_launch(a, pq, early, early, st);
            if (e == cudaErrorNotSupported) return MNB_ERR_UNSUPPORTED;
        }
    }
    if (e != cudaSuccess) return MNB_ERR_CUDA;
    h->last_route = p.route;
    return MNB_OK;
}

int mnb_sync_status(mnb_handle h, void* stream) {
    if (!h) return MNB_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MNB_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, mnb::g_status, sizeof(v)) != cudaSuccess) return MNB_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(mnb::g_status, &zero, sizeof(zero)) != cudaSuccess) return MNB_ERR_CUDA;
    // a wait that gave up may have left an adapter exchange part way: start them afresh
    if ((v & mnb::kStatusTimeout) && mnb::decode_reset_exchange() != cudaSuccess) return MNB_ERR_CUDA;
    return (v & mnb::kStatusTimeout) ? MNB_ERR_DEVICE_TIMEOUT : MNB_OK;
}

const char* mnb_status_str(int code) {
    switch (code) {
        case MNB_OK: return "MNB_OK";
        case MNB_ERR_ARG: return "MNB_ERR_ARG: invalid argument";
        case MNB_ERR_UNSUPPORTED: return "MNB_ERR_UNSUPPORTED: unsupported bits/block/K/rank";
        case MNB_ERR_ALIGN: return "MNB_ERR_ALIGN: pointer not 16-byte aligned";
        case MNB_ERR_CUDA: return "MNB_ERR_CUDA: CUDA runtime error";
        case MNB_ERR_DEVICE_TIMEOUT: return "MNB_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
        case MNB_ERR_NO_DEVICE: return "MNB_ERR_NO_DEVICE: no sm_100-family GPU is current";
        default: return "MNB_ERR_UNKNOWN";
    }
}

int mnb_dequant(const void* Wq, const void* scales, const void* zp, int64_t N, int64_t K, int32_t bits,
                int32_t block_size, void* W16, int32_t variant, void* stream) {
    if (N < 0 || K < 0 || variant < 0 || variant > 1) return MNB_ERR_ARG;
    if (bits != 2 && bits != 4 && bits != 8) return MNB_ERR_UNSUPPORTED;
    if (block_size != 32 || K % (bits == 2 ? 64 : 32) != 0) return MNB_ERR_UNSUPPORTED;
    if (N > INT32_MAX || K > INT32_MAX / 2) return MNB_ERR_UNSUPPORTED;
    if (N == 0 || K == 0) return MNB_OK;
    if (!Wq || !scales || !W16) return MNB_ERR_ARG;
    if (!aligned16(Wq) || !aligned16(scales) || !aligned16(zp) || !aligned16(W16)) return MNB_ERR_ALIGN;
    int sms;
    const int rc = device_setup(&sms);
    if (rc != MNB_OK) return rc;
    const cudaError_t e = mnb::dequant_launch(static_cast<const uint8_t*>(Wq), static_cast<const __half*>(scales),
                                              static_cast<const uint8_t*>(zp), (int)N, (int)K, bits,
                                              static_cast<__half*>(W16), variant,
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MNB_OK : MNB_ERR_CUDA;
}

int mnb_lora_down(const void* X, const void* A, void* T, int64_t Mt, int64_t K, int32_t rank, void* stream) {
    if (Mt < 0 || K < 0) return MNB_ERR_ARG;
    if (rank != 32 || K % 32 != 0) return MNB_ERR_UNSUPPORTED;
    if (Mt > INT32_MAX || K > INT32_MAX / 2) return MNB_ERR_UNSUPPORTED;
    if (Mt == 0) return MNB_OK;
    if (!T) return MNB_ERR_ARG;
    if (!aligned16(X) || !aligned16(A) || !aligned16(T)) return MNB_ERR_ALIGN;
    int sms;
    const int rc = device_setup(&sms);
    if (rc != MNB_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        return mnb::fill_zero_launch(static_cast<__half*>(T), (size_t)Mt * 32, st) == cudaSuccess ? MNB_OK
                                                                                                   : MNB_ERR_CUDA;
    }
    if (!X || !A) return MNB_ERR_ARG;
    const cudaError_t e = mnb::lora_down_launch(static_cast<const __half*>(X), static_cast<const __half*>(A),
                                                static_cast<__half*>(T), (int)Mt, (int)K, false, st);
    return e == cudaSuccess ? MNB_OK : MNB_ERR_CUDA;
}

}  // extern "C"
