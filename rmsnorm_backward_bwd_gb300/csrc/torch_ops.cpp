// Differentiable RMSNorm, fused-add RMSNorm and LayerNorm as PyTorch
// operators written in C++ over the library's C ABI
// (include/rmsnorm_gb300.h). Built into its own shared library next to the
// CUDA library and loaded with torch.ops.load_library; it links against the
// CUDA library and calls nothing but its exported functions.
//
// Two layers, registered with the PyTorch dispatcher in namespace rn_gb300:
//   - raw calls (rmsnorm_fwd, rmsnorm_bwd, fused_add_rmsnorm_fwd,
//     fused_add_rmsnorm_bwd, layernorm_fwd, layernorm_bwd), CUDA only:
//     argument checks, outputs and workspace from the caching allocator, and
//     one C-ABI call on the input's device and current stream.
//   - differentiable ops (rmsnorm, fused_add_rmsnorm, layernorm): C++
//     autograd functions that flatten to [M, N], save what the backward
//     needs and call the raw calls through the dispatcher. The autograd
//     engine runs their backward on its device thread without entering
//     Python.
//
// What is saved and returned follows FlyDSL PR #800 ("Add fused-add /
// residual backward", sections "Summary" and "What's included"): the forward
// saves the per-row fp32 rstd and the backward consumes it; the fused-add
// variant returns (out, residual_out), saves residual_out (= x + residual,
// the tensor the statistic is taken of) and returns one gradient for both x
// and residual. LayerNorm saves the per-row mean and rstd (issue #769, plan
// "PR 5 -- LayerNorm backward").
#include <ATen/ATen.h>
#include <c10/cuda/CUDAGuard.h>
#include <c10/cuda/CUDAStream.h>
#include <torch/csrc/autograd/custom_function.h>
#include <torch/library.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "../../include/rmsnorm_gb300.h"

namespace {

using at::Tensor;
using torch::autograd::AutogradContext;
using torch::autograd::tensor_list;

// ------------------------------------------------------------ argument checks

int dtype_code(const Tensor &t) {
    switch (t.scalar_type()) {
    case at::kFloat: return RN_F32;
    case at::kHalf: return RN_F16;
    case at::kBFloat16: return RN_BF16;
    default: break;
    }
    TORCH_CHECK_TYPE(false, "unsupported dtype ", t.scalar_type(), " (f32, f16, bf16 only)");
    return -1;
}

// A CUDA tensor on ref's device, of dtype dt, contiguous, optionally of `shape`.
void need(const char *name, const Tensor &t, const Tensor &ref, at::ScalarType dt,
          c10::IntArrayRef shape = {}, bool check_shape = false) {
    TORCH_CHECK_VALUE(t.defined(), name, " is required");
    TORCH_CHECK_VALUE(t.is_cuda(), name, " is on ", t.device(),
                      ": these ops run on CUDA devices only");
    TORCH_CHECK_VALUE(t.device() == ref.device(), name, " is on ", t.device(), ", expected ",
                      ref.device());
    TORCH_CHECK_VALUE(t.scalar_type() == dt, "dtype mismatch: ", name, " is ", t.scalar_type(),
                      ", expected ", dt);
    TORCH_CHECK_VALUE(t.is_contiguous(), name, " must be contiguous");
    if (check_shape)
        TORCH_CHECK_VALUE(t.sizes() == shape, name, " has shape ", t.sizes(), ", expected ",
                          shape);
}

// Rows and width of x for a weight of shape [N]: M = numel / N.
std::pair<int64_t, int64_t> rows_of(const Tensor &x, const Tensor &w) {
    TORCH_CHECK_VALUE(x.dim() >= 1, "input must have at least one dimension");
    const int64_t N = x.size(-1);
    TORCH_CHECK_VALUE(w.dim() == 1 && w.size(0) == N, "weight has shape ", w.sizes(),
                      ", expected (", N, ",)");
    return {N ? x.numel() / N : 0, N};
}

void check(rn_status st, const char *call) {
    if (st == RN_OK) return;
    if (st == RN_ERR_INVALID_ARG)
        TORCH_CHECK_VALUE(false, call, ": ", rn_status_string(st), ": ", rn_last_error());
    TORCH_CHECK(false, call, ": ", rn_status_string(st), ": ", rn_last_error());
}

void *stream_of(const Tensor &t) {
    return c10::cuda::getCurrentCUDAStream(t.get_device()).stream();
}

Tensor f32_vector(int64_t n, const Tensor &like) {
    return at::empty({n}, like.options().dtype(at::kFloat));
}

// The backward's workspace, kept per (device, stream) so that a call does
// not allocate one each time (calls that share one are ordered on their
// stream). A workspace replaced by a larger one stays allocated: a CUDA
// graph captured on that stream may still use it. The map is never
// destroyed, so no tensor outlives the CUDA context at process exit.
Tensor workspace(size_t bytes, const Tensor &like) {
    struct Cache {
        std::mutex mu;
        std::map<std::pair<int, void *>, Tensor> live;
        std::vector<Tensor> retired;
    };
    static Cache *cache = new Cache();
    const std::pair<int, void *> key{like.get_device(), stream_of(like)};
    std::lock_guard<std::mutex> lk(cache->mu);
    Tensor &ws = cache->live[key];
    if (!ws.defined() || (size_t)ws.numel() < bytes) {
        if (ws.defined()) cache->retired.push_back(ws);
        // the caching allocator's blocks are 512-byte aligned (the library wants 256)
        ws = at::empty({(int64_t)bytes}, like.options().dtype(at::kByte));
    }
    return ws;
}

// ------------------------------------------------------------ raw calls

std::tuple<Tensor, Tensor> rmsnorm_fwd(const Tensor &x, const Tensor &w, double eps) {
    need("x", x, x, x.scalar_type());
    need("weight", w, x, x.scalar_type());
    const auto [M, N] = rows_of(x, w);
    c10::cuda::CUDAGuard guard(x.device());
    Tensor y = at::empty(x.sizes(), x.options());
    Tensor rstd = f32_vector(M, x);
    check(rn_rmsnorm_fwd(x.data_ptr(), w.data_ptr(), (float)eps, y.data_ptr(),
                         rstd.data_ptr<float>(), M, N, dtype_code(x), stream_of(x)),
          "rn_rmsnorm_fwd");
    return {y, rstd};
}

std::tuple<Tensor, Tensor, Tensor> fused_add_rmsnorm_fwd(const Tensor &x, const Tensor &r,
                                                         const Tensor &w, double eps) {
    need("x", x, x, x.scalar_type());
    need("residual", r, x, x.scalar_type(), x.sizes(), true);
    need("weight", w, x, x.scalar_type());
    const auto [M, N] = rows_of(x, w);
    c10::cuda::CUDAGuard guard(x.device());
    Tensor out = at::empty(x.sizes(), x.options());
    Tensor res_out = at::empty(x.sizes(), x.options());
    Tensor rstd = f32_vector(M, x);
    check(rn_fused_add_rmsnorm_fwd(x.data_ptr(), r.data_ptr(), w.data_ptr(), (float)eps,
                                   out.data_ptr(), res_out.data_ptr(), rstd.data_ptr<float>(), M,
                                   N, dtype_code(x), stream_of(x)),
          "rn_fused_add_rmsnorm_fwd");
    return {out, res_out, rstd};
}

// Shared by both RMSNorm backward calls; dres undefined = none.
// Returns (dx, dweight [undefined unless want_cast], dweight_f32 [undefined
// unless want_f32]). Without the fp32 output the library sums the weight
// gradient in its deterministic scratch mode (one launch fewer); without
// either, no weight gradient is computed.
std::tuple<Tensor, Tensor, Tensor> rms_bwd(const Tensor &x, const Tensor &w, const Tensor &dy,
                                           const Tensor &rstd, const Tensor &dres,
                                           bool want_cast, bool fused, bool want_f32) {
    const char *xname = fused ? "added" : "x";
    need(xname, x, x, x.scalar_type());
    need("weight", w, x, x.scalar_type());
    need("dy", dy, x, x.scalar_type(), x.sizes(), true);
    const auto [M, N] = rows_of(x, w);
    need("rstd", rstd, x, at::kFloat, {M}, true);
    if (dres.defined()) need("dresidual_out", dres, x, x.scalar_type(), x.sizes(), true);
    c10::cuda::CUDAGuard guard(x.device());
    const int code = dtype_code(x);
    size_t ws_bytes = 0;
    check(rn_bwd_workspace_bytes(M, N, code, &ws_bytes), "rn_bwd_workspace_bytes");
    Tensor ws = workspace(ws_bytes, x);
    Tensor dx = at::empty(x.sizes(), x.options());
    Tensor dw32 = want_f32 ? f32_vector(N, x) : Tensor();
    Tensor dw = want_cast ? at::empty({N}, x.options()) : Tensor();
    void *dwp = want_cast ? dw.data_ptr() : nullptr;
    float *dw32p = want_f32 ? dw32.data_ptr<float>() : nullptr;
    if (fused)
        check(rn_fused_add_rmsnorm_bwd(x.data_ptr(), w.data_ptr(), dy.data_ptr(),
                                       rstd.data_ptr<float>(),
                                       dres.defined() ? dres.data_ptr() : nullptr, dx.data_ptr(),
                                       dw32p, dwp, ws.data_ptr(), ws_bytes, M, N, code,
                                       stream_of(x)),
              "rn_fused_add_rmsnorm_bwd");
    else
        check(rn_rmsnorm_bwd(x.data_ptr(), w.data_ptr(), dy.data_ptr(), rstd.data_ptr<float>(),
                             dx.data_ptr(), dw32p, dwp, ws.data_ptr(), ws_bytes, M, N, code,
                             stream_of(x)),
              "rn_rmsnorm_bwd");
    return {dx, dw, dw32};
}

std::tuple<Tensor, Tensor, Tensor> rmsnorm_bwd(const Tensor &x, const Tensor &w, const Tensor &dy,
                                               const Tensor &rstd, bool want_cast, bool want_f32) {
    return rms_bwd(x, w, dy, rstd, Tensor(), want_cast, false, want_f32);
}

std::tuple<Tensor, Tensor, Tensor> fused_add_rmsnorm_bwd(const Tensor &added, const Tensor &w,
                                                         const Tensor &dy, const Tensor &rstd,
                                                         const c10::optional<Tensor> &dres,
                                                         bool want_cast, bool want_f32) {
    return rms_bwd(added, w, dy, rstd, dres.has_value() ? *dres : Tensor(), want_cast, true,
                   want_f32);
}

std::tuple<Tensor, Tensor, Tensor> layernorm_fwd(const Tensor &x, const Tensor &w,
                                                 const c10::optional<Tensor> &b, double eps) {
    need("x", x, x, x.scalar_type());
    need("weight", w, x, x.scalar_type());
    const auto [M, N] = rows_of(x, w);
    const bool has_b = b.has_value() && b->defined();
    if (has_b) need("bias", *b, x, x.scalar_type(), {N}, true);
    c10::cuda::CUDAGuard guard(x.device());
    Tensor y = at::empty(x.sizes(), x.options());
    Tensor mean = f32_vector(M, x), rstd = f32_vector(M, x);
    check(rn_layernorm_fwd(x.data_ptr(), w.data_ptr(), has_b ? b->data_ptr() : nullptr,
                           (float)eps, y.data_ptr(), mean.data_ptr<float>(),
                           rstd.data_ptr<float>(), M, N, dtype_code(x), stream_of(x)),
          "rn_layernorm_fwd");
    return {y, mean, rstd};
}

// Returns (dx, dgamma, dbeta, dgamma_f32, dbeta_f32); the casts are
// undefined unless want_cast, the fp32 sums unless want_f32, the dbeta pair
// unless want_dbeta.
std::tuple<Tensor, Tensor, Tensor, Tensor, Tensor> layernorm_bwd(
    const Tensor &x, const Tensor &w, const Tensor &dy, const Tensor &mean, const Tensor &rstd,
    bool want_dbeta, bool want_cast, bool want_f32) {
    need("x", x, x, x.scalar_type());
    need("weight", w, x, x.scalar_type());
    need("dy", dy, x, x.scalar_type(), x.sizes(), true);
    const auto [M, N] = rows_of(x, w);
    need("mean", mean, x, at::kFloat, {M}, true);
    need("rstd", rstd, x, at::kFloat, {M}, true);
    c10::cuda::CUDAGuard guard(x.device());
    const int code = dtype_code(x);
    size_t ws_bytes = 0;
    check(rn_layernorm_bwd_workspace_bytes(M, N, code, &ws_bytes),
          "rn_layernorm_bwd_workspace_bytes");
    Tensor ws = workspace(ws_bytes, x);
    Tensor dx = at::empty(x.sizes(), x.options());
    Tensor dg32 = want_f32 ? f32_vector(N, x) : Tensor();
    Tensor db32 = want_f32 && want_dbeta ? f32_vector(N, x) : Tensor();
    Tensor dg = want_cast ? at::empty({N}, x.options()) : Tensor();
    Tensor db = want_cast && want_dbeta ? at::empty({N}, x.options()) : Tensor();
    check(rn_layernorm_bwd(x.data_ptr(), w.data_ptr(), dy.data_ptr(), mean.data_ptr<float>(),
                           rstd.data_ptr<float>(), dx.data_ptr(),
                           dg32.defined() ? dg32.data_ptr<float>() : nullptr,
                           db32.defined() ? db32.data_ptr<float>() : nullptr,
                           dg.defined() ? dg.data_ptr() : nullptr,
                           db.defined() ? db.data_ptr() : nullptr, ws.data_ptr(), ws_bytes, M, N,
                           code, stream_of(x)),
          "rn_layernorm_bwd");
    return {dx, dg, db, dg32, db32};
}

// ------------------------------------------------------------ autograd layer

// The raw calls through the dispatcher (so that any backend registered for
// them serves the differentiable ops). Callers hold a
// BelowAutograd guard: the raw calls have no autograd formula, and the
// dispatcher then goes straight to the backend kernel.
using BelowAutograd = at::AutoDispatchBelowADInplaceOrView;

template <typename Sig>
c10::TypedOperatorHandle<Sig> raw(const char *name) {
    return c10::Dispatcher::singleton().findSchemaOrThrow(name, "").template typed<Sig>();
}

Tensor rows2d(const Tensor &t, int64_t N) { return t.reshape({-1, N}).contiguous(); }

int64_t width(const Tensor &x) {
    TORCH_CHECK_VALUE(x.dim() >= 1, "input must have at least one dimension");
    return x.size(-1);
}

struct RMSNormFunction : public torch::autograd::Function<RMSNormFunction> {
    static Tensor forward(AutogradContext *ctx, const Tensor &x, const Tensor &w, double eps) {
        static auto op = raw<std::tuple<Tensor, Tensor>(const Tensor &, const Tensor &, double)>(
            "rn_gb300::rmsnorm_fwd");
        const Tensor x2 = rows2d(x, width(x));
        const Tensor wc = w.contiguous();
        auto [y, rstd] = op.call(x2, wc, eps);
        ctx->save_for_backward({x2, wc, rstd});
        ctx->saved_data["shape"] = x.sizes().vec();
        return y.view(x.sizes());
    }

    static tensor_list backward(AutogradContext *ctx, tensor_list grads) {
        static auto op = raw<std::tuple<Tensor, Tensor, Tensor>(const Tensor &, const Tensor &,
                                                                const Tensor &, const Tensor &,
                                                                bool, bool)>(
            "rn_gb300::rmsnorm_bwd");
        BelowAutograd below;
        const auto saved = ctx->get_saved_variables();
        const bool need_x = ctx->needs_input_grad(0), need_w = ctx->needs_input_grad(1);
        if (!(need_x || need_w)) return {Tensor(), Tensor(), Tensor()};
        const Tensor &x2 = saved[0];
        // an fp32 weight takes the fp32 sum itself (no cast launch); a 16-bit one only the
        // cast (no fp32 output: the deterministic two-launch path); none when the weight
        // needs no gradient
        const bool f32 = x2.scalar_type() == at::kFloat;
        auto [dx, dw, dw32] = op.call(x2, saved[1], rows2d(grads[0], x2.size(1)), saved[2],
                                      need_w && !f32, need_w && f32);
        const auto shape = ctx->saved_data["shape"].toIntVector();
        return {need_x ? dx.view(shape) : Tensor(), need_w ? (f32 ? dw32 : dw) : Tensor(),
                Tensor()};
    }
};

struct FusedAddRMSNormFunction : public torch::autograd::Function<FusedAddRMSNormFunction> {
    static tensor_list forward(AutogradContext *ctx, const Tensor &x, const Tensor &r,
                               const Tensor &w, double eps) {
        static auto op = raw<std::tuple<Tensor, Tensor, Tensor>(const Tensor &, const Tensor &,
                                                                const Tensor &, double)>(
            "rn_gb300::fused_add_rmsnorm_fwd");
        TORCH_CHECK_VALUE(r.sizes() == x.sizes(), "residual has shape ", r.sizes(),
                          ", expected ", x.sizes());
        const int64_t N = width(x);
        const Tensor wc = w.contiguous();
        auto [out, res_out, rstd] = op.call(rows2d(x, N), rows2d(r, N), wc, eps);
        ctx->save_for_backward({res_out, wc, rstd});
        ctx->saved_data["shape"] = x.sizes().vec();
        // an output whose gradient autograd does not produce stays undefined:
        // no zero tensor is made for residual_out when only `out` is used
        ctx->set_materialize_grads(false);
        return {out.view(x.sizes()), res_out.view(x.sizes())};
    }

    static tensor_list backward(AutogradContext *ctx, tensor_list grads) {
        static auto op = raw<std::tuple<Tensor, Tensor, Tensor>(
            const Tensor &, const Tensor &, const Tensor &, const Tensor &,
            const c10::optional<Tensor> &, bool, bool)>("rn_gb300::fused_add_rmsnorm_bwd");
        BelowAutograd below;
        const auto saved = ctx->get_saved_variables();
        const bool need_x = ctx->needs_input_grad(0), need_r = ctx->needs_input_grad(1),
                   need_w = ctx->needs_input_grad(2);
        const tensor_list none = {Tensor(), Tensor(), Tensor(), Tensor()};
        if (!(need_x || need_r || need_w)) return none;
        const Tensor &added = saved[0];
        const int64_t N = added.size(1);
        Tensor d_out = grads[0];
        const Tensor &d_res = grads[1];
        if (!d_out.defined()) {
            if (!d_res.defined()) return none;
            // only residual_out was used: out's gradient is zero
            d_out = at::zeros_like(added);
        }
        c10::optional<Tensor> dres;
        if (d_res.defined()) dres = rows2d(d_res, N);
        const bool f32 = added.scalar_type() == at::kFloat;
        auto [dx, dw, dw32] = op.call(added, saved[1], rows2d(d_out, N), saved[2], dres,
                                      need_w && !f32, need_w && f32);
        const auto shape = ctx->saved_data["shape"].toIntVector();
        const Tensor g = dx.view(shape);
        return {need_x ? g : Tensor(), need_r ? g : Tensor(),
                need_w ? (f32 ? dw32 : dw) : Tensor(), Tensor()};
    }
};

struct LayerNormFunction : public torch::autograd::Function<LayerNormFunction> {
    // Without a bias, b is an empty optional: it is then no variable input
    // of the node, which has two input edges (x, weight) instead of three.
    static Tensor forward(AutogradContext *ctx, const Tensor &x, const Tensor &w,
                          const c10::optional<Tensor> &b, double eps) {
        static auto op = raw<std::tuple<Tensor, Tensor, Tensor>(
            const Tensor &, const Tensor &, const c10::optional<Tensor> &, double)>(
            "rn_gb300::layernorm_fwd");
        const Tensor x2 = rows2d(x, width(x));
        const Tensor wc = w.contiguous();
        const bool has_b = b.has_value() && b->defined();
        c10::optional<Tensor> bc;
        if (has_b) bc = b->contiguous();
        auto [y, mean, rstd] = op.call(x2, wc, bc, eps);
        ctx->save_for_backward({x2, wc, mean, rstd});
        ctx->saved_data["shape"] = x.sizes().vec();
        ctx->saved_data["has_bias"] = has_b;
        return y.view(x.sizes());
    }

    static tensor_list backward(AutogradContext *ctx, tensor_list grads) {
        static auto op = raw<std::tuple<Tensor, Tensor, Tensor, Tensor, Tensor>(
            const Tensor &, const Tensor &, const Tensor &, const Tensor &, const Tensor &, bool,
            bool, bool)>("rn_gb300::layernorm_bwd");
        BelowAutograd below;
        const auto saved = ctx->get_saved_variables();
        const bool need_x = ctx->needs_input_grad(0), need_w = ctx->needs_input_grad(1);
        const bool need_b = ctx->saved_data["has_bias"].toBool() && ctx->needs_input_grad(2);
        if (!(need_x || need_w || need_b)) return {Tensor(), Tensor(), Tensor(), Tensor()};
        const Tensor &x2 = saved[0];
        const bool f32 = x2.scalar_type() == at::kFloat;
        auto [dx, dg, db, dg32, db32] = op.call(x2, saved[1], rows2d(grads[0], x2.size(1)),
                                                saved[2], saved[3], need_b,
                                                (need_w || need_b) && !f32,
                                                (need_w || need_b) && f32);
        const auto shape = ctx->saved_data["shape"].toIntVector();
        return {need_x ? dx.view(shape) : Tensor(), need_w ? (f32 ? dg32 : dg) : Tensor(),
                need_b ? (f32 ? db32 : db) : Tensor(), Tensor()};
    }
};

Tensor rmsnorm(const Tensor &x, const Tensor &w, double eps) {
    return RMSNormFunction::apply(x, w, eps);
}

std::tuple<Tensor, Tensor> fused_add_rmsnorm(const Tensor &x, const Tensor &r, const Tensor &w,
                                             double eps) {
    auto outs = FusedAddRMSNormFunction::apply(x, r, w, eps);
    return {outs[0], outs[1]};
}

Tensor layernorm(const Tensor &x, const Tensor &w, const c10::optional<Tensor> &b, double eps) {
    c10::optional<Tensor> bias;
    if (b.has_value() && b->defined()) bias = *b;
    return LayerNormFunction::apply(x, w, bias, eps);
}

}  // namespace

TORCH_LIBRARY(rn_gb300, m) {
    m.def("rmsnorm_fwd(Tensor x, Tensor weight, float eps) -> (Tensor, Tensor)");
    m.def("rmsnorm_bwd(Tensor x, Tensor weight, Tensor dy, Tensor rstd, bool want_cast, "
          "bool want_f32=True) -> (Tensor, Tensor, Tensor)");
    m.def("fused_add_rmsnorm_fwd(Tensor x, Tensor residual, Tensor weight, float eps) "
          "-> (Tensor, Tensor, Tensor)");
    m.def("fused_add_rmsnorm_bwd(Tensor added, Tensor weight, Tensor dy, Tensor rstd, "
          "Tensor? dresidual_out, bool want_cast, bool want_f32=True) -> (Tensor, Tensor, Tensor)");
    m.def("layernorm_fwd(Tensor x, Tensor weight, Tensor? bias, float eps) "
          "-> (Tensor, Tensor, Tensor)");
    m.def("layernorm_bwd(Tensor x, Tensor weight, Tensor dy, Tensor mean, Tensor rstd, "
          "bool want_dbeta, bool want_cast, bool want_f32=True) "
          "-> (Tensor, Tensor, Tensor, Tensor, Tensor)");
    m.def("rmsnorm(Tensor x, Tensor weight, float eps) -> Tensor");
    m.def("fused_add_rmsnorm(Tensor x, Tensor residual, Tensor weight, float eps) "
          "-> (Tensor, Tensor)");
    m.def("layernorm(Tensor x, Tensor weight, Tensor? bias, float eps) -> Tensor");
}

TORCH_LIBRARY_IMPL(rn_gb300, CUDA, m) {
    m.impl("rmsnorm_fwd", rmsnorm_fwd);
    m.impl("rmsnorm_bwd", rmsnorm_bwd);
    m.impl("fused_add_rmsnorm_fwd", fused_add_rmsnorm_fwd);
    m.impl("fused_add_rmsnorm_bwd", fused_add_rmsnorm_bwd);
    m.impl("layernorm_fwd", layernorm_fwd);
    m.impl("layernorm_bwd", layernorm_bwd);
}

// The raw calls are not differentiable (their outputs carry no gradient
// history, as with the C ABI itself): skip the autograd key for them rather
// than run PyTorch's generic not-implemented fallback on every call.
TORCH_LIBRARY_IMPL(rn_gb300, Autograd, m) {
    for (const char *name : {"rmsnorm_fwd", "rmsnorm_bwd", "fused_add_rmsnorm_fwd",
                             "fused_add_rmsnorm_bwd", "layernorm_fwd", "layernorm_bwd"})
        m.impl(name, torch::CppFunction::makeFallthrough());
}

TORCH_LIBRARY_IMPL(rn_gb300, CompositeImplicitAutograd, m) {
    m.impl("rmsnorm", rmsnorm);
    m.impl("fused_add_rmsnorm", fused_add_rmsnorm);
    m.impl("layernorm", layernorm);
}
