// abi.cu -- the extern "C" entry points of libssm_gb300 (declared in
// include/ssm_gb300.h): host-side argument validation, TMA descriptor
// encoding, workspace layout and kernel launches.  Nothing here allocates
// device memory; every buffer belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "conv_args.cuh"
#include "decode_args.cuh"
#include "gemm_args.cuh"
#include "host_util.h"
#include "scan_args.cuh"
#include "ssm_gb300.h"

namespace ssm_host {

thread_local int g_last_cuda_error = 0;

ssm_status fail_cuda(cudaError_t e, ssm_status s) {
    g_last_cuda_error = static_cast<int>(e);
    return s;
}

// ---- device check: the kernels are built for sm_103a only
ssm_status check_device() {
    static std::mutex mu;
    static int cached[64];   // 0 unknown, 1 ok, 2 wrong arch
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, SSM_ERR_DEVICE);
    if (dev < 0 || dev >= 64) return SSM_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return fail_cuda(e, SSM_ERR_DEVICE);
        cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return cached[dev] == 1 ? SSM_OK : SSM_ERR_DEVICE;
}

// ---- TMA descriptors, encoded through the runtime's driver entry point (the
// library does not link libcuda, so it loads on machines without a driver).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace ssm_host

namespace {

using ssm_host::aligned16;
using ssm_host::align256;
using ssm_host::check_device;
using ssm_host::encode_fn;
using ssm_host::fail_cuda;
using ssm_host::g_last_cuda_error;

// (M, dinner) activation viewed as [batch][seqlen][dinner] with row stride ld;
// box = box_ch channels x box_rows steps x 1 batch row; out-of-range reads fill 0.
bool encode_act(CUtensorMap* m, const void* ptr, int dtype, int dinner, int seqlen, int batch,
                int64_t ld, int box_rows, int box_ch = 32) {
    auto fn = encode_fn();
    if (!fn) return false;
    const size_t es = dtype == SSM_BF16 ? 2 : 4;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(dinner), static_cast<cuuint64_t>(seqlen),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * es,
                             static_cast<cuuint64_t>(ld) * es * static_cast<cuuint64_t>(seqlen)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_ch), static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(m, dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---- descriptor validation
struct Lds {
    int64_t u, delta, z, B, C, out, dout, du, ddelta, dz, dB, dC;
};

int64_t pick(int64_t ld, int64_t packed) { return ld == 0 ? packed : ld; }

ssm_status validate(const ssm_scan_desc* d, Lds& r) {
    if (!d) return SSM_ERR_NULL;
    if (d->batch < 0 || d->seqlen < 0 || d->dinner < 0 || d->dstate < 0 ||
        d->dstate > SSM_MAX_DSTATE)
        return SSM_ERR_SHAPE;
    if (d->dtype != SSM_F32 && d->dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (d->disc != SSM_DISC_EULER && d->disc != SSM_DISC_ZOH) return SSM_ERR_DTYPE;
    const int64_t D = d->dinner, N = d->dstate;
    r.u = pick(d->ld_u, D);
    r.delta = pick(d->ld_delta, D);
    r.z = pick(d->ld_z, D);
    r.out = pick(d->ld_out, D);
    r.dout = pick(d->ld_dout, D);
    r.du = pick(d->ld_du, D);
    r.ddelta = pick(d->ld_ddelta, D);
    r.dz = pick(d->ld_dz, D);
    r.B = pick(d->ld_B, N);
    r.C = pick(d->ld_C, N);
    r.dB = pick(d->ld_dB, N);
    r.dC = pick(d->ld_dC, N);
    const int64_t acts[] = {r.u, r.delta, r.z, r.out, r.dout, r.du, r.ddelta, r.dz};
    for (int64_t v : acts)
        if (v < D || v > (int64_t(1) << 31)) return SSM_ERR_SHAPE;
    const int64_t bcs[] = {r.B, r.C, r.dB, r.dC};
    for (int64_t v : bcs)
        if (v < N || v > (int64_t(1) << 31)) return SSM_ERR_SHAPE;
    // every flat index must fit comfortably in 64 bits and TMA coordinates in
    // int32; batch rows map to the grid's y dimension (at most 65535)
    if (static_cast<int64_t>(d->batch) * d->seqlen > (int64_t(1) << 40)) return SSM_ERR_SHAPE;
    if (d->batch > 65535) return SSM_ERR_SHAPE;
    const int64_t es = d->dtype == SSM_BF16 ? 2 : 4;
    if ((D * es) % 16 != 0) return SSM_ERR_ALIGN;
    for (int64_t v : acts)
        if ((v * es) % 16 != 0) return SSM_ERR_ALIGN;
    return SSM_OK;
}

int nt_of(int dstate) { return dstate <= 8 ? 8 : 16; }
int64_t nchunks_of(int seqlen) { return (static_cast<int64_t>(seqlen) + ssm::kChunk - 1) / ssm::kChunk; }
int64_t nck_of(int seqlen) { return seqlen > 0 ? nchunks_of(seqlen) - 1 : 0; }

// Saved context: fp32 checkpoints [batch][nck][NT][dinner], then the pre-gate
// y (M, dinner) in the activation dtype (read by the backward for dz).
size_t ctx_ck_bytes(const ssm_scan_desc* d) {
    return static_cast<size_t>(d->batch) * nck_of(d->seqlen) * nt_of(d->dstate) * d->dinner *
           sizeof(float);
}
size_t ctx_y_offset(const ssm_scan_desc* d) { return align256(ctx_ck_bytes(d)); }
size_t ctx_total_bytes(const ssm_scan_desc* d) {
    const size_t es = d->dtype == SSM_BF16 ? 2 : 4;
    return ctx_y_offset(d) + static_cast<size_t>(d->batch) * d->seqlen * d->dinner * es;
}

bool encode_ck(CUtensorMap* m, const void* ptr, int dinner, int64_t rows, int nt, int box_ch) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(dinner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(dinner) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_ch), static_cast<cuuint32_t>(nt)};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (M, dstate) B or C viewed as [batch][seqlen][dstate]; box = NT states x
// box_rows steps (states past dstate read as 0).
bool encode_bc(CUtensorMap* m, const void* ptr, int dtype, int dstate, int seqlen, int batch,
               int64_t ld, int nt, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const size_t es = dtype == SSM_BF16 ? 2 : 4;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(dstate), static_cast<cuuint64_t>(seqlen),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * es,
                             static_cast<cuuint64_t>(ld) * es * static_cast<cuuint64_t>(seqlen)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(nt), static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
              3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B and C travel by TMA when both rows start on 16-byte boundaries; otherwise
// the kernels read them with plain loads.
bool bc_tma_ok(const ssm_scan_desc* d, const void* B, const void* C, int64_t ldB, int64_t ldC) {
    const int64_t es = d->dtype == SSM_BF16 ? 2 : 4;
    return d->dstate > 0 && B && C && aligned16(B) && aligned16(C) && (ldB * es) % 16 == 0 &&
           (ldC * es) % 16 == 0;
}

struct BwdLayout {
    int cw, ncl, nseg, seg_chunks;
    size_t off_cg, off_cdl, off_sg, off_sds, off_sd0;
    size_t off_bc, off_dA, off_dD, total;
};

// Forward workspace: the time-segment buffers (none with one segment).
struct FwdLayout {
    int nseg, seg_tiles;
    size_t off_h0, off_segh, off_segds, total;
};
FwdLayout fwd_layout(const ssm_scan_desc* d) {
    FwdLayout l{};
    const int g = ssm::fwd_segments(d->batch, d->dinner, d->seqlen);
    l.seg_tiles = ssm::fwd_seg_tiles(d->seqlen, g);
    const int ntiles = (d->seqlen + ssm::kFwdTile - 1) / ssm::kFwdTile;
    l.nseg = l.seg_tiles > 0 ? (ntiles + l.seg_tiles - 1) / l.seg_tiles : 1;
    if (l.nseg <= 1) {
        l.nseg = 1;
        l.seg_tiles = ntiles > 0 ? ntiles : 1;
        return l;
    }
    const size_t NT = nt_of(d->dstate);
    const size_t hb = static_cast<size_t>(d->batch) * l.nseg * NT * d->dinner * sizeof(float);
    l.off_h0 = 0;
    l.off_segh = align256(hb);
    l.off_segds = l.off_segh + align256(hb);
    l.total = l.off_segds + align256(static_cast<size_t>(d->batch) * l.nseg * d->dinner * sizeof(float));
    return l;
}

BwdLayout bwd_layout(const ssm_scan_desc* d) {
    BwdLayout l{};
    l.cw = ssm::bwd_channels(d->batch, d->dinner);
    l.ncl = static_cast<int>((static_cast<int64_t>(d->dinner) + l.cw - 1) / l.cw);
    const size_t M = static_cast<size_t>(d->batch) * d->seqlen;
    const size_t NT = nt_of(d->dstate);
    const int nchunks = static_cast<int>(nchunks_of(d->seqlen));
    const int g = ssm::bwd_segments(d->batch, d->dinner, d->seqlen, l.cw);
    l.seg_chunks = nchunks > 0 ? (nchunks + g - 1) / g : 1;
    l.nseg = nchunks > 0 ? (nchunks + l.seg_chunks - 1) / l.seg_chunks : 1;
    const size_t planes = static_cast<size_t>(d->batch) * l.nseg;   // dA / dD partial planes
    l.off_bc = 0;
    l.off_dA = align256(static_cast<size_t>(l.ncl) * M * 2 * NT * sizeof(float));
    l.off_dD = l.off_dA + align256(planes * d->dinner * NT * sizeof(float));
    size_t end = l.off_dD + align256(planes * d->dinner * sizeof(float));
    if (l.nseg > 1) {
        const size_t gs = align256(planes * NT * d->dinner * sizeof(float));
        const size_t ds = align256(planes * d->dinner * sizeof(float));
        l.off_cg = end;
        l.off_sg = l.off_cg + gs;
        l.off_cdl = l.off_sg + gs;
        l.off_sds = l.off_cdl + ds;
        l.off_sd0 = l.off_sds + ds;
        end = l.off_sd0 + ds;
    }
    l.total = end;
    return l;
}

}  // namespace

extern "C" {

size_t ssm_scan_ctx_bytes(const ssm_scan_desc* d) {
    Lds r;
    if (validate(d, r) != SSM_OK) return 0;
    return ctx_total_bytes(d);
}

size_t ssm_scan_fwd_workspace_bytes(const ssm_scan_desc* d) {
    Lds r;
    if (validate(d, r) != SSM_OK) return 0;
    return fwd_layout(d).total;
}

size_t ssm_scan_bwd_workspace_bytes(const ssm_scan_desc* d) {
    Lds r;
    if (validate(d, r) != SSM_OK) return 0;
    return bwd_layout(d).total;
}

}  // extern "C"

namespace ssm_host {

// The forward behind ssm_scan_fwd (h_init = h_last = null), ssm_scan_fwd_state
// (ctx = null) and the block's prefill.
ssm_status scan_fwd_impl(const ssm_scan_desc* d, const void* u, const void* delta_raw,
                         const float* A_log, const void* B, const void* C, const float* D,
                         const void* z, void* out, void* ctx, size_t ctx_bytes, const float* h_init,
                         float* h_last, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Lds r;
    ssm_status st = validate(d, r);
    if (st != SSM_OK) return st;
    const int64_t M = static_cast<int64_t>(d->batch) * d->seqlen;
    const size_t hbytes = static_cast<size_t>(d->batch) * d->dstate * d->dinner * sizeof(float);
    if (h_init && h_last && hbytes > 0) {
        const char *i0 = reinterpret_cast<const char*>(h_init), *l0 = reinterpret_cast<const char*>(h_last);
        if (i0 < l0 + hbytes && l0 < i0 + hbytes) return SSM_ERR_SHAPE;   // the two states overlap
    }
    if ((h_init && (reinterpret_cast<uintptr_t>(h_init) & 3u)) ||
        (h_last && (reinterpret_cast<uintptr_t>(h_last) & 3u)))
        return SSM_ERR_ALIGN;
    if (M == 0 && h_last && hbytes > 0) {
        // no step: the final state is the initial one
        if ((st = check_device()) != SSM_OK) return st;
        cudaError_t e = h_init ? cudaMemcpyAsync(h_last, h_init, hbytes, cudaMemcpyDeviceToDevice, stream)
                               : cudaMemsetAsync(h_last, 0, hbytes, stream);
        return e == cudaSuccess ? SSM_OK : fail_cuda(e);
    }
    if (M == 0 || d->dinner == 0) return SSM_OK;
    if (!u || !delta_raw || !out) return SSM_ERR_NULL;
    if (d->dstate > 0 && (!B || !C || !A_log)) return SSM_ERR_NULL;
    if (!aligned16(u) || !aligned16(delta_raw) || !aligned16(out) || (z && !aligned16(z)))
        return SSM_ERR_ALIGN;
    if (ctx) {
        if (ctx_bytes < ssm_scan_ctx_bytes(d)) return SSM_ERR_WORKSPACE;
        if (!aligned16(ctx)) return SSM_ERR_ALIGN;
    }
    const FwdLayout fl = fwd_layout(d);
    if (fl.total > 0) {
        if (!workspace || workspace_bytes < fl.total) return SSM_ERR_WORKSPACE;
        if (!aligned16(workspace)) return SSM_ERR_ALIGN;
    }
    if ((st = check_device()) != SSM_OK) return st;

    ssm::FwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const int nt = nt_of(d->dstate);
    const bool bct = bc_tma_ok(d, B, C, r.B, r.C);
    const int fc = ssm::kFwdChannels;
    if (!encode_act(&maps.u, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u, ssm::kFwdTile, fc) ||
        !encode_act(&maps.dr, delta_raw, d->dtype, d->dinner, d->seqlen, d->batch, r.delta,
                    ssm::kFwdTile, fc) ||
        !encode_act(&maps.z, z ? z : u, d->dtype, d->dinner, d->seqlen, d->batch, z ? r.z : r.u,
                    ssm::kFwdTile, fc) ||
        !(bct ? encode_bc(&maps.B, B, d->dtype, d->dstate, d->seqlen, d->batch, r.B, nt, ssm::kFwdTile)
              : encode_act(&maps.B, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u, ssm::kFwdTile)) ||
        !(bct ? encode_bc(&maps.C, C, d->dtype, d->dstate, d->seqlen, d->batch, r.C, nt, ssm::kFwdTile)
              : encode_act(&maps.C, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u, ssm::kFwdTile)) ||
        !encode_act(&maps.out, out, d->dtype, d->dinner, d->seqlen, d->batch, r.out, ssm::kFwdTile, fc))
        return SSM_ERR_DEVICE;
    if (ctx) {
        // saved pre-gate y (packed) and the chunk-boundary states
        if (!encode_act(&maps.y, static_cast<char*>(ctx) + ctx_y_offset(d), d->dtype, d->dinner, d->seqlen,
                        d->batch, d->dinner, ssm::kFwdTile, fc))
            return SSM_ERR_DEVICE;
        const int64_t ck_rows = static_cast<int64_t>(d->batch) * nck_of(d->seqlen) * nt;
        if (ck_rows > 0 && !encode_ck(&maps.ck, ctx, d->dinner, ck_rows, nt, fc)) return SSM_ERR_DEVICE;
    }
    ssm::ScanFwdArgs a{};
    a.B = B;
    a.C = C;
    a.A_log = A_log;
    a.D = D;
    a.out = out;
    a.ctx = static_cast<float*>(ctx);
    a.ysave = ctx ? static_cast<char*>(ctx) + ctx_y_offset(d) : nullptr;
    a.batch = d->batch;
    a.seqlen = d->seqlen;
    a.dinner = d->dinner;
    a.dstate = d->dstate;
    a.ld_B = r.B;
    a.ld_C = r.C;
    a.ld_out = r.out;
    a.nck = static_cast<int>(nck_of(d->seqlen));
    a.bc_tma = bct ? 1 : 0;
    a.nseg = fl.nseg;
    a.seg_tiles = fl.seg_tiles;
    if (fl.nseg > 1) {
        char* w = static_cast<char*>(workspace);
        a.h0 = reinterpret_cast<float*>(w + fl.off_h0);
        a.seg_h = reinterpret_cast<float*>(w + fl.off_segh);
        a.seg_ds = reinterpret_cast<float*>(w + fl.off_segds);
    }
    a.h_init = h_init;
    a.h_last = h_last;
    cudaError_t e = ssm::launch_scan_fwd(d->dtype, nt, d->disc, z != nullptr, maps, a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

}  // namespace ssm_host

extern "C" {

ssm_status ssm_scan_fwd(const ssm_scan_desc* d, const void* u, const void* delta_raw,
                        const float* A_log, const void* B, const void* C, const float* D,
                        const void* z, void* out, void* ctx, size_t ctx_bytes, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    return ssm_host::scan_fwd_impl(d, u, delta_raw, A_log, B, C, D, z, out, ctx, ctx_bytes, nullptr, nullptr,
                         workspace, workspace_bytes, stream);
}

ssm_status ssm_scan_fwd_state(const ssm_scan_desc* d, const void* u, const void* delta_raw,
                              const float* A_log, const void* B, const void* C, const float* D,
                              const void* z, void* out, const float* h_init, float* h_last,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return ssm_host::scan_fwd_impl(d, u, delta_raw, A_log, B, C, D, z, out, nullptr, 0, h_init, h_last,
                         workspace, workspace_bytes, stream);
}

ssm_status ssm_scan_bwd(const ssm_scan_desc* d, const void* u, const void* delta_raw,
                        const float* A_log, const void* B, const void* C, const float* D,
                        const void* z, const void* dout, const void* ctx, size_t ctx_bytes,
                        void* du, void* ddelta_raw, float* dA_log, void* dB, void* dC, float* dD,
                        void* dz, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Lds r;
    ssm_status st = validate(d, r);
    if (st != SSM_OK) return st;
    const int64_t M = static_cast<int64_t>(d->batch) * d->seqlen;
    const bool any_work = M > 0 && d->dinner > 0;
    const bool any_out = (M > 0 && d->dstate > 0) || (d->dinner > 0);
    if (!any_out) return SSM_OK;
    if (any_work) {
        if (!u || !delta_raw || !dout || !du || !ddelta_raw) return SSM_ERR_NULL;
        if (z && !dz) return SSM_ERR_NULL;
        if (!aligned16(u) || !aligned16(delta_raw) || !aligned16(dout) || !aligned16(du) ||
            !aligned16(ddelta_raw) || (z && !aligned16(z)) || (dz && !aligned16(dz)))
            return SSM_ERR_ALIGN;
        if (nck_of(d->seqlen) > 0 || z) {
            if (!ctx) return SSM_ERR_NULL;
            if (ctx_bytes < ssm_scan_ctx_bytes(d)) return SSM_ERR_WORKSPACE;
            if (!aligned16(ctx)) return SSM_ERR_ALIGN;
        }
    }
    if (d->dinner > 0 && d->dstate > 0 && !A_log) return SSM_ERR_NULL;
    if (d->dinner > 0 && d->dstate > 0 && !dA_log) return SSM_ERR_NULL;
    if (M > 0 && d->dstate > 0 && (!B || !C || !dB || !dC)) return SSM_ERR_NULL;
    const BwdLayout lay = bwd_layout(d);
    if (workspace_bytes < lay.total || (lay.total > 0 && !workspace)) return SSM_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return SSM_ERR_ALIGN;
    if ((st = check_device()) != SSM_OK) return st;

    char* ws = static_cast<char*>(workspace);
    const int nt = nt_of(d->dstate);
    if (any_work) {
        ssm::BwdMaps maps;
        const int64_t nck = nck_of(d->seqlen);
        const bool bct = bc_tma_ok(d, B, C, r.B, r.C);
        const bool ysaved = z != nullptr && ctx != nullptr;
        const void* ybuf = ysaved ? static_cast<const char*>(ctx) + ctx_y_offset(d) : u;
        const int bc = lay.cw;
        if (!encode_act(&maps.u, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u, ssm::kChunk, bc) ||
            !encode_act(&maps.dr, delta_raw, d->dtype, d->dinner, d->seqlen, d->batch, r.delta,
                        ssm::kChunk, bc) ||
            !encode_act(&maps.dout, dout, d->dtype, d->dinner, d->seqlen, d->batch, r.dout,
                        ssm::kChunk, bc) ||
            !encode_act(&maps.z, z ? z : u, d->dtype, d->dinner, d->seqlen, d->batch, z ? r.z : r.u,
                        ssm::kChunk, bc) ||
            !encode_act(&maps.y, ybuf, d->dtype, d->dinner, d->seqlen, d->batch,
                        ysaved ? d->dinner : r.u, ssm::kChunk, bc) ||
            !(nck > 0 ? encode_ck(&maps.ck, ctx, d->dinner, static_cast<int64_t>(d->batch) * nck * nt, nt, bc)
                      : encode_act(&maps.ck, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u,
                                   ssm::kChunk, bc)) ||
            !(bct ? encode_bc(&maps.B, B, d->dtype, d->dstate, d->seqlen, d->batch, r.B, nt, ssm::kChunk)
                  : encode_act(&maps.B, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u, ssm::kChunk)) ||
            !(bct ? encode_bc(&maps.C, C, d->dtype, d->dstate, d->seqlen, d->batch, r.C, nt, ssm::kChunk)
                  : encode_act(&maps.C, u, d->dtype, d->dinner, d->seqlen, d->batch, r.u, ssm::kChunk)))
            return SSM_ERR_DEVICE;
        ssm::ScanBwdArgs a{};
        a.B = B;
        a.C = C;
        a.A_log = A_log;
        a.D = D;
        a.du = du;
        a.ddelta = ddelta_raw;
        a.dz = dz;
        a.ws_bc = reinterpret_cast<float*>(ws + lay.off_bc);
        a.ws_dA = reinterpret_cast<float*>(ws + lay.off_dA);
        a.ws_dD = reinterpret_cast<float*>(ws + lay.off_dD);
        a.nseg = lay.nseg;
        a.seg_chunks = lay.seg_chunks;
        if (lay.nseg > 1) {
            a.carry_g = reinterpret_cast<float*>(ws + lay.off_cg);
            a.seg_g = reinterpret_cast<float*>(ws + lay.off_sg);
            a.carry_dl = reinterpret_cast<float*>(ws + lay.off_cdl);
            a.seg_ds = reinterpret_cast<float*>(ws + lay.off_sds);
            a.seg_d0 = reinterpret_cast<float*>(ws + lay.off_sd0);
        }
        a.batch = d->batch;
        a.seqlen = d->seqlen;
        a.dinner = d->dinner;
        a.dstate = d->dstate;
        a.ld_B = r.B;
        a.ld_C = r.C;
        a.ld_du = r.du;
        a.ld_ddelta = r.ddelta;
        a.ld_dz = r.dz;
        a.nck = static_cast<int>(nck_of(d->seqlen));
        a.ncl = lay.ncl;
        a.cw = lay.cw;
        a.bc_tma = bct ? 1 : 0;
        cudaError_t e = ssm::launch_scan_bwd(d->dtype, nt, d->disc, z != nullptr, maps, a, stream);
        if (e != cudaSuccess) return fail_cuda(e);
    }
    ssm::ScanReduceArgs ra{};
    ra.ws_bc = reinterpret_cast<const float*>(ws + lay.off_bc);
    ra.ws_dA = reinterpret_cast<const float*>(ws + lay.off_dA);
    ra.ws_dD = reinterpret_cast<const float*>(ws + lay.off_dD);
    ra.A_log = A_log;
    ra.dB = dB;
    ra.dC = dC;
    ra.dA_log = dA_log;
    ra.dD = dD;
    ra.batch = d->batch;
    ra.seqlen = d->seqlen;
    ra.dinner = d->dinner;
    ra.dstate = d->dstate;
    ra.nt = nt;
    ra.ncl = any_work ? lay.ncl : 0;
    ra.nb_sum = any_work ? d->batch * lay.nseg : 0;
    ra.ld_dB = r.dB;
    ra.ld_dC = r.dC;
    ra.is_bf16 = d->dtype == SSM_BF16;
    cudaError_t e = ssm::launch_scan_reduce(ra, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

ssm_status ssm_scan_step(const ssm_scan_desc* d, const void* u, const void* delta_raw,
                         const float* A_log, const void* B, const void* C, const float* D,
                         const void* z, float* h, void* out, cudaStream_t stream) {
    Lds r;
    ssm_status st = validate(d, r);
    if (st != SSM_OK) return st;
    if (d->seqlen != 1) return SSM_ERR_SHAPE;
    if (d->batch == 0 || d->dinner == 0) return SSM_OK;
    if (!u || !delta_raw || !out) return SSM_ERR_NULL;
    if (d->dstate > 0 && (!B || !C || !A_log || !h)) return SSM_ERR_NULL;
    if (!aligned16(u) || !aligned16(delta_raw) || !aligned16(out) || (z && !aligned16(z)) ||
        (d->dstate > 0 && !aligned16(h)))
        return SSM_ERR_ALIGN;
    if ((st = check_device()) != SSM_OK) return st;
    ssm::ScanStepArgs a{};
    a.u = u;
    a.dr = delta_raw;
    a.z = z;
    a.B = B;
    a.C = C;
    a.A_log = A_log;
    a.D = D;
    a.h = h;
    a.out = out;
    a.batch = d->batch;
    a.dinner = d->dinner;
    a.dstate = d->dstate;
    a.ld_u = r.u;
    a.ld_dr = r.delta;
    a.ld_z = r.z;
    a.ld_B = r.B;
    a.ld_C = r.C;
    a.ld_out = r.out;
    cudaError_t e = ssm::launch_scan_step(d->dtype, nt_of(d->dstate), d->disc, z != nullptr, a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

ssm_status ssm_conv1d_silu_step(int32_t batch, int32_t dinner, int32_t kconv, const float* x,
                                int64_t ld_x, const float* w, const float* bias, float* conv_state,
                                float* out, int64_t ld_out, cudaStream_t stream) {
    if (batch < 0 || dinner < 0 || kconv < 1 || kconv > 8) return SSM_ERR_SHAPE;
    ld_x = ld_x ? ld_x : dinner;
    ld_out = ld_out ? ld_out : dinner;
    if (ld_x < dinner || ld_out < dinner) return SSM_ERR_SHAPE;
    if (batch == 0 || dinner == 0) return SSM_OK;
    if (!x || !w || !out || (kconv > 1 && !conv_state)) return SSM_ERR_NULL;
    if (dinner % 4 || ld_x % 4 || ld_out % 4 || !aligned16(x) || !aligned16(out) ||
        (kconv > 1 && !aligned16(conv_state)) || (bias && !aligned16(bias)))
        return SSM_ERR_ALIGN;
    ssm_status st = check_device();
    if (st != SSM_OK) return st;
    ssm::ConvStepArgs a{};
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.state = conv_state;
    a.out = out;
    a.batch = batch;
    a.dinner = dinner;
    a.kconv = kconv;
    a.ld_x = ld_x;
    a.ld_out = ld_out;
    cudaError_t e = ssm::launch_conv_step(a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

ssm_status ssm_conv1d_state_from_prompt(int32_t batch, int32_t seqlen, int32_t dinner,
                                        int32_t kconv, const float* x, int64_t ld_x,
                                        float* conv_state, cudaStream_t stream) {
    if (batch < 0 || seqlen < 0 || dinner < 0 || kconv < 1 || kconv > 8) return SSM_ERR_SHAPE;
    ld_x = ld_x ? ld_x : dinner;
    if (ld_x < dinner) return SSM_ERR_SHAPE;
    if (batch == 0 || dinner == 0 || kconv == 1) return SSM_OK;
    if (!conv_state || (seqlen > 0 && !x)) return SSM_ERR_NULL;
    if (dinner % 4 || ld_x % 4 || (x && !aligned16(x)) || !aligned16(conv_state)) return SSM_ERR_ALIGN;
    ssm_status st = check_device();
    if (st != SSM_OK) return st;
    ssm::ConvStateFillArgs a{};
    a.x = x;
    a.state = conv_state;
    a.batch = batch;
    a.seqlen = seqlen;
    a.dinner = dinner;
    a.kconv = kconv;
    a.ld_x = ld_x;
    cudaError_t e = ssm::launch_conv_state_fill(a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

ssm_status ssm_conv1d_silu(int32_t batch, int32_t seqlen, int32_t dinner, int32_t kconv,
                           const float* x, int64_t ld_x, const float* w, const float* bias,
                           float* out, int64_t ld_out, cudaStream_t stream) {
    if (batch < 0 || seqlen < 0 || dinner < 0 || kconv < 1 || kconv > 8) return SSM_ERR_SHAPE;
    ld_x = ld_x ? ld_x : dinner;
    ld_out = ld_out ? ld_out : dinner;
    if (ld_x < dinner || ld_out < dinner) return SSM_ERR_SHAPE;
    if (static_cast<int64_t>(batch) * seqlen == 0 || dinner == 0) return SSM_OK;
    if (!x || !w || !out) return SSM_ERR_NULL;
    if (dinner % 4 || ld_x % 4 || ld_out % 4 || !aligned16(x) || !aligned16(out) ||
        (bias && !aligned16(bias)))
        return SSM_ERR_ALIGN;
    ssm_status st = check_device();
    if (st != SSM_OK) return st;
    ssm::ConvArgs a{};
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.out = out;
    a.batch = batch;
    a.seqlen = seqlen;
    a.dinner = dinner;
    a.kconv = kconv;
    a.ld_x = ld_x;
    a.ld_out = ld_out;
    cudaError_t e = ssm::launch_conv1d_fwd(a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

size_t ssm_conv1d_silu_bwd_workspace_bytes(int32_t batch, int32_t seqlen, int32_t dinner,
                                           int32_t kconv) {
    if (batch < 0 || seqlen < 0 || dinner < 0 || kconv < 1 || kconv > 8) return 0;
    return ssm::conv1d_bwd_workspace_bytes(batch, seqlen, dinner, kconv);
}

ssm_status ssm_conv1d_silu_bwd(int32_t batch, int32_t seqlen, int32_t dinner, int32_t kconv,
                               const float* x, int64_t ld_x, const float* w, const float* bias,
                               const float* dout, int64_t ld_dout, float* dx, int64_t ld_dx,
                               float* dw, float* dbias, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    if (batch < 0 || seqlen < 0 || dinner < 0 || kconv < 1 || kconv > 8) return SSM_ERR_SHAPE;
    ld_x = ld_x ? ld_x : dinner;
    ld_dout = ld_dout ? ld_dout : dinner;
    ld_dx = ld_dx ? ld_dx : dinner;
    if (ld_x < dinner || ld_dout < dinner || ld_dx < dinner) return SSM_ERR_SHAPE;
    if (dinner == 0) return SSM_OK;
    if (!w || !dw) return SSM_ERR_NULL;
    const bool rows = static_cast<int64_t>(batch) * seqlen > 0;
    if (rows && (!x || !dout || !dx)) return SSM_ERR_NULL;
    if (dinner % 4 || ld_x % 4 || ld_dout % 4 || ld_dx % 4 || (x && !aligned16(x)) ||
        (dout && !aligned16(dout)) || (dx && !aligned16(dx)) || (bias && !aligned16(bias)))
        return SSM_ERR_ALIGN;
    const size_t need = ssm::conv1d_bwd_workspace_bytes(batch, seqlen, dinner, kconv);
    if (workspace_bytes < need || (need && !workspace)) return SSM_ERR_WORKSPACE;
    ssm_status st = check_device();
    if (st != SSM_OK) return st;
    ssm::ConvArgs a{};
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.dout = dout;
    a.dx = dx;
    a.dw = dw;
    a.dbias = dbias;
    a.ws = static_cast<float*>(workspace);
    a.batch = batch;
    a.seqlen = seqlen;
    a.dinner = dinner;
    a.kconv = kconv;
    a.ld_x = ld_x;
    a.ld_dout = ld_dout;
    a.ld_dx = ld_dx;
    cudaError_t e = ssm::launch_conv1d_bwd(a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

ssm_status ssm_conv1d_silu_bwd_noalloc(int32_t batch, int32_t seqlen, int32_t dinner,
                                       int32_t kconv, const float* x, int64_t ld_x,
                                       const float* w, const float* bias, const float* dout,
                                       int64_t ld_dout, float* dx, int64_t ld_dx, float* dw,
                                       float* dbias, cudaStream_t stream) {
    if (batch < 0 || seqlen < 0 || dinner < 0 || kconv < 1 || kconv > 8) return SSM_ERR_SHAPE;
    ld_x = ld_x ? ld_x : dinner;
    ld_dout = ld_dout ? ld_dout : dinner;
    ld_dx = ld_dx ? ld_dx : dinner;
    if (ld_x < dinner || ld_dout < dinner || ld_dx < dinner) return SSM_ERR_SHAPE;
    if (dinner == 0) return SSM_OK;
    if (!w || !dw) return SSM_ERR_NULL;
    const bool rows = static_cast<int64_t>(batch) * seqlen > 0;
    if (rows && (!x || !dout || !dx)) return SSM_ERR_NULL;
    if (dinner % 4 || ld_x % 4 || ld_dout % 4 || ld_dx % 4 || (x && !aligned16(x)) ||
        (dout && !aligned16(dout)) || (dx && !aligned16(dx)) || (bias && !aligned16(bias)))
        return SSM_ERR_ALIGN;
    const size_t need = ssm::conv1d_bwd_workspace_bytes(batch, seqlen, dinner, kconv);
    if (need > ssm::kConvNoAllocScratchFloats * sizeof(float)) return SSM_ERR_WORKSPACE;
    ssm_status st = check_device();
    if (st != SSM_OK) return st;
    float* scratch = nullptr;
    cudaError_t e = ssm::conv1d_noalloc_scratch(&scratch);
    if (e != cudaSuccess) return fail_cuda(e, SSM_ERR_DEVICE);
    ssm::ConvArgs a{};
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.dout = dout;
    a.dx = dx;
    a.dw = dw;
    a.dbias = dbias;
    a.ws = scratch;
    a.batch = batch;
    a.seqlen = seqlen;
    a.dinner = dinner;
    a.kconv = kconv;
    a.ld_x = ld_x;
    a.ld_dout = ld_dout;
    a.ld_dx = ld_dx;
    e = ssm::launch_conv1d_bwd(a, stream);
    return e == cudaSuccess ? SSM_OK : fail_cuda(e);
}

const char* ssm_status_string(ssm_status s) {
    switch (s) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "required pointer is NULL";
        case SSM_ERR_SHAPE: return "size or stride out of range";
        case SSM_ERR_ALIGN: return "pointer or row stride breaks the 16-byte alignment rule";
        case SSM_ERR_DTYPE: return "unknown dtype or discretisation";
        case SSM_ERR_WORKSPACE: return "context or workspace too small";
        case SSM_ERR_LAUNCH: return "kernel launch failed";
        case SSM_ERR_DEVICE: return "current device is not an sm_103 GPU";
    }
    return "unknown status";
}

int ssm_last_cuda_error(void) { return g_last_cuda_error; }

int ssm_abi_version(void) { return SSM_GB300_ABI_VERSION; }

unsigned ssm_device_faults(void) {
    unsigned f1 = 0, f2 = 0, f3 = 0, f4 = 0;
    if (check_device() != SSM_OK) return 0;
    ssm::read_clear_fault_fwd(&f1);
    ssm::read_clear_fault_bwd(&f2);
    ssm::read_clear_fault_gemm(&f3);
    ssm::read_clear_fault_probe(&f4);
    return f1 | f2 | f3 | f4;
}

}  // extern "C"
