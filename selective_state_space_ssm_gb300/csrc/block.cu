// block.cu -- extern "C" entry points of the whole Mamba-1 block
// (mamba1_cpu.ts mamba1CpuForward steps 1-11 and mamba1CpuBackward steps
// 11-1; linear and RMSNorm as cpu_ops.ts defines them).  Host-side
// orchestration only: every step runs in this library's kernels (RMSNorm,
// operand transposes, tcgen05 GEMM, conv1d+SiLU, selective scan, column sums), in
// stream order on the caller's stream, in caller-owned memory.
#include <algorithm>
#include <cstring>

#include "gemm_args.cuh"
#include "host_util.h"
#include "ssm_gb300.h"

namespace {

using ssm_host::align256;
using ssm_host::aligned16;
using ssm_host::check_device;
using ssm_host::encode_fn;
using ssm_host::fail_cuda;

constexpr float kRmsEps = 1e-6f;   // cpu_ops.ts RMSNORM_EPS

int64_t round4(int64_t n) { return (n + 3) & ~static_cast<int64_t>(3); }

// Byte offsets of one buffer layout (each region 256-byte aligned).
struct Carve {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    }
};

struct Dims {
    int64_t M;
    int B, L, Dm, D, N, R, K, P, disc;
};

ssm_status check_desc(const ssm_block_desc* d, Dims& s) {
    if (!d) return SSM_ERR_NULL;
    if (d->disc != SSM_DISC_EULER && d->disc != SSM_DISC_ZOH) return SSM_ERR_DTYPE;
    if (d->batch < 0 || d->seqlen < 0 || d->dmodel <= 0 || d->dinner <= 0 || d->dstate <= 0 ||
        d->dstate > SSM_MAX_DSTATE || d->dtrank <= 0 || d->dconv < 1 || d->dconv > 8)
        return SSM_ERR_SHAPE;
    if (d->dmodel % 4 || d->dinner % 4 || d->dstate % 4 || d->dtrank % 4) return SSM_ERR_ALIGN;
    s.B = d->batch;
    s.L = d->seqlen;
    s.M = static_cast<int64_t>(d->batch) * d->seqlen;
    if (s.M > (int64_t(1) << 30)) return SSM_ERR_SHAPE;
    s.Dm = d->dmodel;
    s.D = d->dinner;
    s.N = d->dstate;
    s.R = d->dtrank;
    s.K = d->dconv;
    s.P = d->dtrank + 2 * d->dstate;
    s.disc = d->disc;
    return SSM_OK;
}

ssm_scan_desc scan_desc_of(const Dims& s) {
    ssm_scan_desc sd;
    std::memset(&sd, 0, sizeof(sd));
    sd.batch = s.B;
    sd.seqlen = s.L;
    sd.dinner = s.D;
    sd.dstate = s.N;
    sd.dtype = SSM_F32;
    sd.disc = s.disc;
    sd.ld_u = s.D;
    sd.ld_delta = s.D;
    sd.ld_z = 2 * s.D;
    sd.ld_B = s.P;
    sd.ld_C = s.P;
    sd.ld_out = s.D;
    sd.ld_dout = s.D;
    sd.ld_du = s.D;
    sd.ld_ddelta = s.D;
    sd.ld_dz = 2 * s.D;
    sd.ld_dB = s.P;
    sd.ld_dC = s.P;
    return sd;
}

// Saved activations of the forward.
struct Ctx {
    size_t xn, inv, xz, u, xd, draw, g, scan, total;
};
Ctx ctx_layout(const Dims& s) {
    const size_t f = sizeof(float), M = static_cast<size_t>(s.M);
    Carve c;
    Ctx x;
    x.xn = c.take(M * s.Dm * f);
    x.inv = c.take(M * f);
    x.xz = c.take(M * 2 * s.D * f);
    x.u = c.take(M * s.D * f);
    x.xd = c.take(M * s.P * f);
    x.draw = c.take(M * s.D * f);
    x.g = c.take(M * s.D * f);
    ssm_scan_desc sd = scan_desc_of(s);
    x.scan = c.take(ssm_scan_ctx_bytes(&sd));
    x.total = c.off;
    return x;
}

// Scratch shared by forward and backward (regions reused in stream order).
struct Ws {
    size_t a_hi, b_hi, w_hi;                              // copies of GEMM operands (transposed / aligned)
    size_t dg, du, ddelta, dxd, dxz, dxn;                 // backward activations
    size_t scan, conv, red, scanf, part, part_floats, total;
};
Ws ws_layout(const Dims& s) {
    const size_t f = sizeof(float);
    const int64_t ldM = round4(s.M);
    const int64_t wide = round4(std::max({int64_t(2) * s.D, int64_t(s.Dm), int64_t(s.P), int64_t(s.R)}));
    const int64_t deep = round4(std::max({int64_t(s.D), int64_t(s.R), int64_t(s.Dm)}));
    auto wsz = [](int64_t rows, int64_t cols) {
        return static_cast<size_t>(std::max(rows * round4(cols), cols * round4(rows)));
    };
    const size_t wmax = std::max({wsz(2 * s.D, s.Dm), wsz(s.P, s.D), wsz(s.D, s.R), wsz(s.Dm, s.D)});
    const size_t M = static_cast<size_t>(s.M);
    Carve c;
    Ws w;
    w.a_hi = c.take(static_cast<size_t>(ldM * wide) * f);
    w.b_hi = c.take(static_cast<size_t>(ldM * deep) * f);
    w.w_hi = c.take(wmax * f);
    w.dg = c.take(M * s.D * f);
    w.du = c.take(M * s.D * f);
    w.ddelta = c.take(M * s.D * f);
    w.dxd = c.take(M * s.P * f);
    w.dxz = c.take(M * 2 * s.D * f);
    w.dxn = c.take(M * s.Dm * f);
    ssm_scan_desc sd = scan_desc_of(s);
    w.scan = c.take(ssm_scan_bwd_workspace_bytes(&sd));
    w.conv = c.take(ssm_conv1d_silu_bwd_workspace_bytes(s.B, s.L, s.D, s.K));
    const int rows = static_cast<int>(s.M);
    const size_t red = std::max({ssm::colsum_ws_floats(rows, 2 * s.D), ssm::colsum_ws_floats(rows, s.Dm),
                                 ssm::colsum_ws_floats(rows, s.P), ssm::rmsnorm_ws_floats(rows, s.Dm)});
    w.red = c.take(std::max<size_t>(red, 1) * f);
    w.scanf = c.take(ssm_scan_fwd_workspace_bytes(&sd));
    // split-K partial sums of the GEMMs with few output tiles
    const size_t biggest = std::max({M * 2 * s.D, M * static_cast<size_t>(s.Dm), M * static_cast<size_t>(s.P),
                                     static_cast<size_t>(2) * s.D * s.Dm, static_cast<size_t>(s.P) * s.D,
                                     static_cast<size_t>(s.D) * s.R});
    w.part_floats = std::min<size_t>(size_t(8) << 20, 4 * biggest);
    w.part = c.take(w.part_floats * f);
    w.total = c.off;
    return w;
}

// One GEMM operand: a K-major (rows, cols) fp32 matrix with row stride ld
// (16-byte aligned base and row stride, as TMA needs).
struct Op {
    const float* p;
    int rows, cols;
    int64_t ld;
};

bool encode_op(CUtensorMap* m, const Op& o) {
    const float* p = o.p;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(o.cols), static_cast<cuuint64_t>(o.rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(o.ld) * sizeof(float)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(ssm::kGemmBK), static_cast<cuuint32_t>(ssm::kGemmBM)};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stream-ordered step list of one call; the first failure sticks.
struct Run {
    cudaStream_t st;
    float* part = nullptr;        // split-K partial sums (null: no split)
    size_t part_floats = 0;
    ssm_status status = SSM_OK;

    bool ok() const { return status == SSM_OK; }
    void cuda(cudaError_t e) {
        if (ok() && e != cudaSuccess) status = fail_cuda(e);
    }
    void check(ssm_status s) {
        if (ok() && s != SSM_OK) status = s;
    }

    // x (rows, cols; stride ldx) as a GEMM operand, transposed or not: used in
    // place when it is K-major and TMA-aligned, else copied (transposed) into buf.
    Op operand(const float* x, int64_t ldx, int rows, int cols, bool transpose, float* buf) {
        if (!transpose && aligned16(x) && (ldx * static_cast<int64_t>(sizeof(float))) % 16 == 0)
            return Op{x, rows, cols, ldx};
        Op o{buf, transpose ? cols : rows, transpose ? rows : cols, 0};
        o.ld = round4(o.cols);
        if (ok()) cuda(ssm::launch_operand_copy(x, ldx, rows, cols, transpose ? 1 : 0, buf, o.ld, st));
        return o;
    }

    // x (rows, cols) transposed into buf as a GEMM operand, with the column sums
    // of x written to colsum from the same pass (ws: colsum_ws_floats floats).
    Op operand_t_colsum(const float* x, int64_t ldx, int rows, int cols, float* buf, float* colsum,
                        float* ws) {
        Op o{buf, cols, rows, 0};
        o.ld = round4(o.cols);
        if (ok()) cuda(ssm::launch_operand_copy_t_colsum(x, ldx, rows, cols, buf, o.ld, colsum, ws, st));
        return o;
    }

    // C (A.rows, B.rows) = A B^T (+ bias) (+ R); A.cols == B.cols.
    void gemm(const Op& A, const Op& B, float* C, int64_t ldc, const float* bias, const float* R,
              int64_t ldr) {
        if (!ok()) return;
        ssm::GemmMaps maps;
        if (!encode_op(&maps.a, A) || !encode_op(&maps.b, B)) {
            status = SSM_ERR_DEVICE;
            return;
        }
        ssm::GemmArgs a{};
        a.C = C;
        a.bias = bias;
        a.R = R;
        a.M = A.rows;
        a.N = B.rows;
        a.K = A.cols;
        a.ldc = ldc;
        a.ldr = ldr;
        a.ksplit = part ? ssm::gemm_ksplit(a.M, a.N, a.K, part_floats) : 1;
        a.part = part;
        cuda(ssm::launch_gemm_tf32x3(maps, a, st));
    }
};

template <class T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <class T>
const T* at(const void* base, size_t off) {
    return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

// Scratch of one decode step of the block (M = batch rows of one position).
struct StepWs {
    size_t xn, inv, xz, u, xd, draw, g, a_hi, w_hi, part, part_floats, total;
};
StepWs step_layout(const Dims& s) {
    const size_t f = sizeof(float), M = static_cast<size_t>(s.M);
    const size_t deep = static_cast<size_t>(round4(std::max({int64_t(s.Dm), int64_t(s.D), int64_t(s.R)})));
    auto wsz = [](int64_t rows, int64_t cols) { return static_cast<size_t>(rows * round4(cols)); };
    const size_t wmax = std::max({wsz(2 * s.D, s.Dm), wsz(s.P, s.D), wsz(s.D, s.R), wsz(s.Dm, s.D)});
    Carve c;
    StepWs w;
    w.xn = c.take(M * s.Dm * f);
    w.inv = c.take(M * f);
    w.xz = c.take(M * 2 * s.D * f);
    w.u = c.take(M * s.D * f);
    w.xd = c.take(M * s.P * f);
    w.draw = c.take(M * s.D * f);
    w.g = c.take(M * s.D * f);
    w.a_hi = c.take(M * deep * f);
    w.w_hi = c.take(wmax * f);
    const size_t biggest = std::max({M * 2 * s.D, M * static_cast<size_t>(s.Dm), M * static_cast<size_t>(s.P),
                                     M * static_cast<size_t>(s.D)});
    w.part_floats = std::min<size_t>(size_t(8) << 20, 4 * biggest);
    w.part = c.take(w.part_floats * f);
    w.total = c.off;
    return w;
}

// The four projection weights as the GEMM reads them -- 16-byte aligned
// copies with rows padded to a multiple of 4 floats -- for decode steps that
// reuse them: in_proj (2 dinner, dmodel), x_proj (dtrank + 2 dstate, dinner),
// dt_proj (dinner, dtrank), out_proj (dmodel, dinner).
struct SplitW {
    size_t hi[4], total;
    int rows[4], cols[4];
};
SplitW split_layout(const Dims& s) {
    SplitW w;
    const int rows[4] = {2 * s.D, s.P, s.D, s.Dm};
    const int cols[4] = {s.Dm, s.D, s.R, s.D};
    Carve c;
    for (int i = 0; i < 4; ++i) {
        w.rows[i] = rows[i];
        w.cols[i] = cols[i];
        const size_t bytes = static_cast<size_t>(rows[i]) * round4(cols[i]) * sizeof(float);
        w.hi[i] = c.take(bytes);
    }
    w.total = c.off;
    return w;
}

bool all_weights(const ssm_block_weights* w) {
    return w && w->in_proj_w && w->in_proj_b && w->conv_w && w->conv_b && w->x_proj_w && w->x_proj_b &&
           w->dt_proj_w && w->dt_proj_b && w->A_log && w->D && w->out_proj_w && w->out_proj_b && w->norm_w;
}
bool all_grads(const ssm_block_grads* g) {
    return g && g->in_proj_w && g->in_proj_b && g->conv_w && g->conv_b && g->x_proj_w && g->x_proj_b &&
           g->dt_proj_w && g->dt_proj_b && g->A_log && g->D && g->out_proj_w && g->out_proj_b && g->norm_w;
}

}  // namespace

extern "C" {

size_t ssm_linear_workspace_bytes(int32_t M, int32_t N, int32_t K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    const size_t f = sizeof(float);
    return align256(static_cast<size_t>(M) * round4(K) * f) +
           align256(static_cast<size_t>(N) * round4(K) * f);
}

ssm_status ssm_linear_fwd(int32_t M, int32_t N, int32_t K, const float* X, int64_t ldx,
                          const float* W, int64_t ldw, const float* bias, const float* R,
                          int64_t ldr, float* Y, int64_t ldy, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return SSM_ERR_SHAPE;
    ldx = ldx ? ldx : K;
    ldw = ldw ? ldw : K;
    ldy = ldy ? ldy : N;
    ldr = ldr ? ldr : N;
    if (ldx < K || ldw < K || ldy < N || (R && ldr < N)) return SSM_ERR_SHAPE;
    if (M == 0 || N == 0) return SSM_OK;
    if (!Y || (K > 0 && (!X || !W))) return SSM_ERR_NULL;
    if (!workspace) return SSM_ERR_NULL;
    if (!aligned16(workspace)) return SSM_ERR_ALIGN;
    if (workspace_bytes < ssm_linear_workspace_bytes(M, N, K)) return SSM_ERR_WORKSPACE;
    ssm_status st = check_device();
    if (st != SSM_OK) return st;
    if (K == 0) return SSM_ERR_SHAPE;
    const size_t f = sizeof(float);
    const size_t xa = align256(static_cast<size_t>(M) * round4(K) * f);
    float* xbuf = static_cast<float*>(workspace);
    float* wbuf = at<float>(workspace, xa);
    Run run{stream};
    Op A = run.operand(X, ldx, M, K, false, xbuf);
    Op B = run.operand(W, ldw, N, K, false, wbuf);
    run.gemm(A, B, Y, ldy, bias, R, ldr);
    return run.status;
}

size_t ssm_block_ctx_bytes(const ssm_block_desc* d) {
    Dims s;
    if (check_desc(d, s) != SSM_OK) return 0;
    return ctx_layout(s).total;
}

size_t ssm_block_workspace_bytes(const ssm_block_desc* d) {
    Dims s;
    if (check_desc(d, s) != SSM_OK) return 0;
    return ws_layout(s).total;
}

}  // extern "C"

namespace {

// The block forward; with conv_state / h non-null it also leaves the states
// after the last position (prefill for ssm_block_step).
ssm_status block_fwd_impl(const ssm_block_desc* d, const float* x, const ssm_block_weights* w, float* out,
                          void* ctx, size_t ctx_bytes, float* conv_state, float* h, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    Dims s;
    ssm_status st = check_desc(d, s);
    if (st != SSM_OK) return st;
    if ((conv_state && !aligned16(conv_state)) || (h && !aligned16(h))) return SSM_ERR_ALIGN;
    if (s.M == 0) {
        // no position: the states of a new sequence are zero
        if (!conv_state && !h) return SSM_OK;
        if ((st = check_device()) != SSM_OK) return st;
        const size_t f = sizeof(float);
        if (conv_state && s.K > 1) {
            cudaError_t e = cudaMemsetAsync(conv_state, 0, size_t(s.B) * (s.K - 1) * s.D * f, stream);
            if (e != cudaSuccess) return fail_cuda(e);
        }
        if (h) {
            cudaError_t e = cudaMemsetAsync(h, 0, size_t(s.B) * s.N * s.D * f, stream);
            if (e != cudaSuccess) return fail_cuda(e);
        }
        return SSM_OK;
    }
    if (!x || !out || !ctx || !workspace || !all_weights(w)) return SSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ctx) || !aligned16(workspace))
        return SSM_ERR_ALIGN;
    const Ctx c = ctx_layout(s);
    const Ws ws = ws_layout(s);
    if (ctx_bytes < c.total || workspace_bytes < ws.total) return SSM_ERR_WORKSPACE;
    if ((st = check_device()) != SSM_OK) return st;

    const int M = static_cast<int>(s.M), Dm = s.Dm, D = s.D, N = s.N, R = s.R, P = s.P;
    float* xn = at<float>(ctx, c.xn);
    float* inv = at<float>(ctx, c.inv);
    float* xz = at<float>(ctx, c.xz);
    float* u = at<float>(ctx, c.u);
    float* xd = at<float>(ctx, c.xd);
    float* draw = at<float>(ctx, c.draw);
    float* g = at<float>(ctx, c.g);
    float* ahi = at<float>(workspace, ws.a_hi);
    float* whi = at<float>(workspace, ws.w_hi);

    Run run{stream, at<float>(workspace, ws.part), ws.part_floats};
    // 1. RMSNorm
    run.cuda(ssm::launch_rmsnorm_fwd(x, w->norm_w, M, Dm, kRmsEps, xn, inv, stream));
    // 2. in_proj (x_in | z)
    {
        Op A = run.operand(xn, Dm, M, Dm, false, ahi);
        Op W = run.operand(w->in_proj_w, Dm, 2 * D, Dm, false, whi);
        run.gemm(A, W, xz, 2 * D, w->in_proj_b, nullptr, 0);
    }
    // 4-5. causal conv1d + SiLU on the x_in columns
    if (run.ok()) run.check(ssm_conv1d_silu(s.B, s.L, D, s.K, xz, 2 * D, w->conv_w, w->conv_b, u, D, stream));
    // 6. x_proj -> (dt | B | C)
    {
        Op A = run.operand(u, D, M, D, false, ahi);
        Op W = run.operand(w->x_proj_w, D, P, D, false, whi);
        run.gemm(A, W, xd, P, w->x_proj_b, nullptr, 0);
    }
    // 7. dt_proj -> delta_raw
    {
        Op A = run.operand(xd, P, M, R, false, ahi);
        Op W = run.operand(w->dt_proj_w, R, D, R, false, whi);
        run.gemm(A, W, draw, D, w->dt_proj_b, nullptr, 0);
    }
    // the conv's state after the last position (its last kconv-1 inputs)
    if (run.ok() && conv_state)
        run.check(ssm_conv1d_state_from_prompt(s.B, s.L, D, s.K, xz, 2 * D, conv_state, stream));
    // 8-9. selective scan with the SiLU(z) gate (and the state after the last position)
    if (run.ok()) {
        ssm_scan_desc sd = scan_desc_of(s);
        run.check(ssm_host::scan_fwd_impl(&sd, u, draw, w->A_log, xd + R, xd + R + N, w->D, xz + D, g,
                                          at<char>(ctx, c.scan), c.total - c.scan, nullptr, h,
                                          at<char>(workspace, ws.scanf), ws.total - ws.scanf, stream));
    }
    // 10-11. out_proj + residual
    {
        Op A = run.operand(g, D, M, D, false, ahi);
        Op W = run.operand(w->out_proj_w, D, Dm, D, false, whi);
        run.gemm(A, W, out, Dm, w->out_proj_b, x, Dm);
    }
    return run.status;
}

}  // namespace

extern "C" {

ssm_status ssm_block_fwd(const ssm_block_desc* d, const float* x, const ssm_block_weights* w,
                         float* out, void* ctx, size_t ctx_bytes, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    return block_fwd_impl(d, x, w, out, ctx, ctx_bytes, nullptr, nullptr, workspace, workspace_bytes,
                          stream);
}

ssm_status ssm_block_fwd_state(const ssm_block_desc* d, const float* x, const ssm_block_weights* w,
                               float* out, void* ctx, size_t ctx_bytes, float* conv_state, float* h,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return block_fwd_impl(d, x, w, out, ctx, ctx_bytes, conv_state, h, workspace, workspace_bytes, stream);
}

size_t ssm_block_weights_split_bytes(const ssm_block_desc* d) {
    Dims s;
    if (check_desc(d, s) != SSM_OK) return 0;
    return split_layout(s).total;
}

ssm_status ssm_block_split_weights(const ssm_block_desc* d, const ssm_block_weights* w, void* split,
                                   size_t split_bytes, cudaStream_t stream) {
    Dims s;
    ssm_status st = check_desc(d, s);
    if (st != SSM_OK) return st;
    if (!split || !all_weights(w)) return SSM_ERR_NULL;
    if (!aligned16(split)) return SSM_ERR_ALIGN;
    const SplitW sw = split_layout(s);
    if (split_bytes < sw.total) return SSM_ERR_WORKSPACE;
    if ((st = check_device()) != SSM_OK) return st;
    const float* src[4] = {w->in_proj_w, w->x_proj_w, w->dt_proj_w, w->out_proj_w};
    Run run{stream};
    for (int i = 0; i < 4; ++i)
        run.cuda(ssm::launch_operand_copy(src[i], sw.cols[i], sw.rows[i], sw.cols[i], 0,
                                          at<float>(split, sw.hi[i]), round4(sw.cols[i]), stream));
    return run.status;
}

size_t ssm_block_step_workspace_bytes(const ssm_block_desc* d) {
    Dims s;
    if (check_desc(d, s) != SSM_OK || s.L != 1) return 0;
    return step_layout(s).total;
}

ssm_status ssm_block_step(const ssm_block_desc* d, const float* x, const ssm_block_weights* w,
                          const void* weights_split, float* conv_state, float* h, float* out,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Dims s;
    ssm_status st = check_desc(d, s);
    if (st != SSM_OK) return st;
    if (s.L != 1) return SSM_ERR_SHAPE;
    if (s.M == 0) return SSM_OK;
    if (!x || !out || !h || !workspace || !all_weights(w) || (s.K > 1 && !conv_state)) return SSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(out) || !aligned16(h) || !aligned16(workspace) ||
        (s.K > 1 && !aligned16(conv_state)))
        return SSM_ERR_ALIGN;
    if (weights_split && !aligned16(weights_split)) return SSM_ERR_ALIGN;
    const StepWs ws = step_layout(s);
    if (workspace_bytes < ws.total) return SSM_ERR_WORKSPACE;
    const SplitW sw = split_layout(s);
    // weight operand i: the caller's prepared copy, or the weight itself
    // (copied into the workspace only if it is not TMA-aligned)
    auto weight = [&](Run& run, int i, const float* W) {
        if (weights_split)
            return Op{at<float>(weights_split, sw.hi[i]), sw.rows[i], sw.cols[i], round4(sw.cols[i])};
        return run.operand(W, sw.cols[i], sw.rows[i], sw.cols[i], false, at<float>(workspace, ws.w_hi));
    };
    if ((st = check_device()) != SSM_OK) return st;

    const int M = static_cast<int>(s.M), Dm = s.Dm, D = s.D, N = s.N, R = s.R, P = s.P;
    float* xn = at<float>(workspace, ws.xn);
    float* inv = at<float>(workspace, ws.inv);
    float* xz = at<float>(workspace, ws.xz);
    float* u = at<float>(workspace, ws.u);
    float* xd = at<float>(workspace, ws.xd);
    float* draw = at<float>(workspace, ws.draw);
    float* g = at<float>(workspace, ws.g);
    float* ahi = at<float>(workspace, ws.a_hi);

    Run run{stream, at<float>(workspace, ws.part), ws.part_floats};
    // 1. RMSNorm
    run.cuda(ssm::launch_rmsnorm_fwd(x, w->norm_w, M, Dm, kRmsEps, xn, inv, stream));
    // 2. in_proj (x_in | z)
    {
        Op A = run.operand(xn, Dm, M, Dm, false, ahi);
        Op W = weight(run, 0, w->in_proj_w);
        run.gemm(A, W, xz, 2 * D, w->in_proj_b, nullptr, 0);
    }
    // 4-5. one position of the causal conv1d + SiLU from the carried conv state
    if (run.ok())
        run.check(ssm_conv1d_silu_step(M, D, s.K, xz, 2 * D, w->conv_w, w->conv_b, conv_state, u, D, stream));
    // 6. x_proj -> (dt | B | C)
    {
        Op A = run.operand(u, D, M, D, false, ahi);
        Op W = weight(run, 1, w->x_proj_w);
        run.gemm(A, W, xd, P, w->x_proj_b, nullptr, 0);
    }
    // 7. dt_proj -> delta_raw
    {
        Op A = run.operand(xd, P, M, R, false, ahi);
        Op W = weight(run, 2, w->dt_proj_w);
        run.gemm(A, W, draw, D, w->dt_proj_b, nullptr, 0);
    }
    // 8-9. one position of the selective scan from the carried state, SiLU(z) gate
    if (run.ok()) {
        ssm_scan_desc sd = scan_desc_of(s);
        run.check(ssm_scan_step(&sd, u, draw, w->A_log, xd + R, xd + R + N, w->D, xz + D, h, g, stream));
    }
    // 10-11. out_proj + residual
    {
        Op A = run.operand(g, D, M, D, false, ahi);
        Op W = weight(run, 3, w->out_proj_w);
        run.gemm(A, W, out, Dm, w->out_proj_b, x, Dm);
    }
    return run.status;
}

ssm_status ssm_block_bwd(const ssm_block_desc* d, const float* x, const ssm_block_weights* w,
                         const float* dout, const void* ctx, size_t ctx_bytes, float* dx,
                         const ssm_block_grads* gr, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    Dims s;
    ssm_status st = check_desc(d, s);
    if (st != SSM_OK) return st;
    if (!all_grads(gr)) return SSM_ERR_NULL;
    if (s.M == 0) {
        // No rows: every gradient is zero.
        if ((st = check_device()) != SSM_OK) return st;
        const size_t f = sizeof(float);
        const int64_t D = s.D, Dm = s.Dm, P = s.P, R = s.R, N = s.N, K = s.K;
        const std::pair<float*, size_t> zs[] = {
            {gr->in_proj_w, 2 * D * Dm}, {gr->in_proj_b, 2 * D}, {gr->conv_w, D * K}, {gr->conv_b, D},
            {gr->x_proj_w, P * D},       {gr->x_proj_b, P},      {gr->dt_proj_w, D * R}, {gr->dt_proj_b, D},
            {gr->A_log, D * N},          {gr->D, D},             {gr->out_proj_w, Dm * D}, {gr->out_proj_b, Dm},
            {gr->norm_w, Dm}};
        for (const auto& z : zs) {
            cudaError_t e = cudaMemsetAsync(z.first, 0, z.second * f, stream);
            if (e != cudaSuccess) return fail_cuda(e);
        }
        return SSM_OK;
    }
    if (!x || !dout || !ctx || !dx || !workspace || !all_weights(w)) return SSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(dout) || !aligned16(ctx) || !aligned16(dx) || !aligned16(workspace))
        return SSM_ERR_ALIGN;
    const Ctx c = ctx_layout(s);
    const Ws ws = ws_layout(s);
    if (ctx_bytes < c.total || workspace_bytes < ws.total) return SSM_ERR_WORKSPACE;
    if ((st = check_device()) != SSM_OK) return st;

    const int M = static_cast<int>(s.M), Dm = s.Dm, D = s.D, N = s.N, R = s.R, P = s.P;
    const float* xn = at<float>(ctx, c.xn);
    const float* inv = at<float>(ctx, c.inv);
    const float* xz = at<float>(ctx, c.xz);
    const float* u = at<float>(ctx, c.u);
    const float* xd = at<float>(ctx, c.xd);
    const float* draw = at<float>(ctx, c.draw);
    const float* g = at<float>(ctx, c.g);
    float* ahi = at<float>(workspace, ws.a_hi);
    float* bhi = at<float>(workspace, ws.b_hi);
    float* whi = at<float>(workspace, ws.w_hi);
    float* dg = at<float>(workspace, ws.dg);
    float* du = at<float>(workspace, ws.du);
    float* ddelta = at<float>(workspace, ws.ddelta);
    float* dxd = at<float>(workspace, ws.dxd);
    float* dxz = at<float>(workspace, ws.dxz);
    float* dxn = at<float>(workspace, ws.dxn);
    float* red = at<float>(workspace, ws.red);

    Run run{stream, at<float>(workspace, ws.part), ws.part_floats};
    // Linear backward of Y = X W^T + b (cpu_ops.ts linearBackward), with
    // dY (rows, nout; stride lddy), X (rows, k; stride ldx), W (nout, k):
    //   dX = dY W  -> dX (stride lddx, + R when accumulate)
    //   dW = dY^T X, db = column sums of dY.
    auto linear_bwd = [&](const float* dY, int64_t lddy, int nout, const float* X, int64_t ldx, int k,
                          const float* W, float* dX, int64_t lddx, bool accumulate, float* dW, float* db) {
        if (dX) {
            Op A = run.operand(dY, lddy, M, nout, false, ahi);
            Op Wt = run.operand(W, k, nout, k, true, whi);   // (k, nout)
            run.gemm(A, Wt, dX, lddx, nullptr, accumulate ? dX : nullptr, lddx);
        }
        Op At = run.operand_t_colsum(dY, lddy, M, nout, ahi, db, red);   // (nout, M); db
        Op Xt = run.operand(X, ldx, M, k, true, bhi);                     // (k, M)
        run.gemm(At, Xt, dW, k, nullptr, nullptr, 0);
    };

    // 10. out_proj (the residual's share of dx is added at step 1)
    linear_bwd(dout, Dm, Dm, g, D, D, w->out_proj_w, dg, D, false, gr->out_proj_w, gr->out_proj_b);
    // 9-8. gate and selective scan: du, ddelta, dB | dC into dxd, dz into dxz
    if (run.ok()) {
        ssm_scan_desc sd = scan_desc_of(s);
        run.check(ssm_scan_bwd(&sd, u, draw, w->A_log, xd + R, xd + R + N, w->D, xz + D, dg,
                               at<char>(ctx, c.scan), c.total - c.scan, du, ddelta, gr->A_log, dxd + R,
                               dxd + R + N, gr->D, dxz + D, at<char>(workspace, ws.scan),
                               ws.conv - ws.scan, stream));
    }
    // 7. dt_proj: d(dt) into the first R columns of dxd
    linear_bwd(ddelta, D, D, xd, P, R, w->dt_proj_w, dxd, P, false, gr->dt_proj_w, gr->dt_proj_b);
    // 6. x_proj: du += dxd W_x
    linear_bwd(dxd, P, P, u, D, D, w->x_proj_w, du, D, true, gr->x_proj_w, gr->x_proj_b);
    // 5-4. SiLU and the causal conv: d(x_in) into the first D columns of dxz
    if (run.ok())
        run.check(ssm_conv1d_silu_bwd(s.B, s.L, D, s.K, xz, 2 * D, w->conv_w, w->conv_b, du, D, dxz, 2 * D,
                                      gr->conv_w, gr->conv_b, at<char>(workspace, ws.conv),
                                      ws.red - ws.conv, stream));
    // 2. in_proj
    linear_bwd(dxz, 2 * D, 2 * D, xn, Dm, Dm, w->in_proj_w, dxn, Dm, false, gr->in_proj_w, gr->in_proj_b);
    // 1. RMSNorm, plus the residual path: dx = dout + d(rmsnorm)
    if (run.ok())
        run.cuda(ssm::launch_rmsnorm_bwd(dxn, x, w->norm_w, inv, dout, M, Dm, dx, gr->norm_w, red, stream));
    (void)N;
    return run.status;
}

}  // extern "C"

// ---- A stack of blocks with activation checkpointing (the pages' model runs
// its layers one after another, each block with its own residual, and its
// backward recomputes every layer's forward from the layer's saved input
// instead of keeping all layers' activations).  Host orchestration over the
// block entry points above: one block context and one block workspace are
// reused by every layer.
namespace {

struct StackWs {
    size_t bctx, bws, tmp, g0, g1, total;
};
StackWs stack_ws_layout(const ssm_block_desc* d, const Dims& s) {
    StackWs l{};
    Carve cv;
    const size_t act = static_cast<size_t>(s.M) * s.Dm * sizeof(float);
    l.bctx = cv.take(ssm_block_ctx_bytes(d));
    l.bws = cv.take(ssm_block_workspace_bytes(d));
    l.tmp = cv.take(act);   // the recomputed forward's output (not needed, but written)
    l.g0 = cv.take(act);    // dL/d(hidden) of alternate layers
    l.g1 = cv.take(act);
    l.total = cv.off;
    return l;
}
size_t stack_ctx_bytes_of(const Dims& s, int layers) {
    return static_cast<size_t>(layers - 1) * align256(static_cast<size_t>(s.M) * s.Dm * sizeof(float));
}
// Input of layer i (> 0): the output of layer i-1, kept in the stack context.
float* stack_hidden(void* ctx, const Dims& s, int i) {
    return reinterpret_cast<float*>(static_cast<char*>(ctx) +
                                    static_cast<size_t>(i - 1) *
                                        align256(static_cast<size_t>(s.M) * s.Dm * sizeof(float)));
}

}  // namespace

extern "C" {

size_t ssm_stack_ctx_bytes(const ssm_block_desc* d, int32_t layers) {
    Dims s;
    if (layers < 1 || check_desc(d, s) != SSM_OK) return 0;
    return stack_ctx_bytes_of(s, layers);
}

size_t ssm_stack_workspace_bytes(const ssm_block_desc* d, int32_t layers) {
    Dims s;
    if (layers < 1 || check_desc(d, s) != SSM_OK) return 0;
    return stack_ws_layout(d, s).total;
}

ssm_status ssm_stack_fwd(const ssm_block_desc* d, int32_t layers, const float* x,
                         const ssm_block_weights* weights, float* out, void* ctx, size_t ctx_bytes,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Dims s;
    ssm_status st = check_desc(d, s);
    if (st != SSM_OK) return st;
    if (layers < 1) return SSM_ERR_SHAPE;
    if (!weights) return SSM_ERR_NULL;
    for (int i = 0; i < layers; ++i)
        if (!all_weights(&weights[i])) return SSM_ERR_NULL;
    if (s.M == 0) return SSM_OK;
    if (!x || !out || !workspace || (layers > 1 && !ctx)) return SSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(out) || !aligned16(workspace) || (ctx && !aligned16(ctx)))
        return SSM_ERR_ALIGN;
    const StackWs l = stack_ws_layout(d, s);
    if (ctx_bytes < stack_ctx_bytes_of(s, layers) || workspace_bytes < l.total) return SSM_ERR_WORKSPACE;
    if ((st = check_device()) != SSM_OK) return st;
    char* w = static_cast<char*>(workspace);
    const float* h = x;
    for (int i = 0; i < layers && st == SSM_OK; ++i) {
        float* o = (i + 1 < layers) ? stack_hidden(ctx, s, i + 1) : out;
        st = ssm_block_fwd(d, h, &weights[i], o, w + l.bctx, l.bws - l.bctx, w + l.bws, l.tmp - l.bws,
                           stream);
        h = o;
    }
    return st;
}

ssm_status ssm_stack_bwd(const ssm_block_desc* d, int32_t layers, const float* x,
                         const ssm_block_weights* weights, const float* dout, const void* ctx,
                         size_t ctx_bytes, float* dx, const ssm_block_grads* grads, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    Dims s;
    ssm_status st = check_desc(d, s);
    if (st != SSM_OK) return st;
    if (layers < 1) return SSM_ERR_SHAPE;
    if (!weights || !grads) return SSM_ERR_NULL;
    for (int i = 0; i < layers; ++i)
        if (!all_weights(&weights[i]) || !all_grads(&grads[i])) return SSM_ERR_NULL;
    if (s.M == 0) {
        // no rows: every gradient is zero (the block backward writes them)
        for (int i = 0; i < layers && st == SSM_OK; ++i)
            st = ssm_block_bwd(d, x, &weights[i], dout, ctx, 0, dx, &grads[i], workspace, 0, stream);
        return st;
    }
    if (!x || !dout || !dx || !workspace || (layers > 1 && !ctx)) return SSM_ERR_NULL;
    if (!aligned16(x) || !aligned16(dout) || !aligned16(dx) || !aligned16(workspace) ||
        (ctx && !aligned16(ctx)))
        return SSM_ERR_ALIGN;
    const StackWs l = stack_ws_layout(d, s);
    if (ctx_bytes < stack_ctx_bytes_of(s, layers) || workspace_bytes < l.total) return SSM_ERR_WORKSPACE;
    if ((st = check_device()) != SSM_OK) return st;
    char* w = static_cast<char*>(workspace);
    void* hidden_ctx = const_cast<void*>(ctx);
    const float* g = dout;   // dL/d(output of the current layer)
    for (int i = layers - 1; i >= 0 && st == SSM_OK; --i) {
        const float* h = i == 0 ? x : stack_hidden(hidden_ctx, s, i);
        // recompute the layer's forward from its saved input, then its backward
        st = ssm_block_fwd(d, h, &weights[i], reinterpret_cast<float*>(w + l.tmp), w + l.bctx,
                           l.bws - l.bctx, w + l.bws, l.tmp - l.bws, stream);
        if (st != SSM_OK) break;
        float* dh = i == 0 ? dx : reinterpret_cast<float*>(w + ((i & 1) ? l.g1 : l.g0));
        st = ssm_block_bwd(d, h, &weights[i], g, w + l.bctx, l.bws - l.bctx, dh, &grads[i], w + l.bws,
                           l.tmp - l.bws, stream);
        g = dh;
    }
    return st;
}

}  // extern "C"
