"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the
fp64 oracle on the same seeded inputs, and compare them.

Tolerance (stated for the operator's floating outputs y and normOut):
|gpu - ref| <= tol * (1 + |ref|) with tol = 1e-2 for bf16 and 2e-3 for fp16
outputs, ref being the oracle's fp64 value. The INT4 pack is compared bit for bit.
"""
import numpy as np
import torch

import oracle

TOL = {torch.bfloat16: 1e-2, torch.float16: 2e-3}


def to_device(prob, device="cuda"):
    for f in ("x1", "x2", "scale", "offset", "bias", "residual", "gamma"):
        v = getattr(prob, f)
        if v is not None:
            setattr(prob, f, v.to(device))
    return prob


def gpu_weight(wq, prob):
    """x2 as the library consumes it: INT4 packed on the GPU by the pack kernel, or INT8."""
    if prob.wbits == 4:
        return wq.pack_int4(prob.x2.to("cuda").contiguous())
    return prob.x2.to("cuda").contiguous()


def run_gpu(wq, prob, kernel=0, w=None, y=None, normOut=None, workspace=None):
    if w is None:
        w = gpu_weight(wq, prob)
    y, no = wq.matmul_add_rmsnorm(prob.x1, w, prob.scale, prob.offset, prob.bias, prob.residual,
                                  prob.gamma, prob.eps, prob.group, y=y, normOut=normOut,
                                  workspace=workspace, kernel=kernel)
    torch.cuda.synchronize()
    return y, no


def sample_rows(M, n_sample, seed=1234):
    if M <= n_sample + 2:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=n_sample, replace=False)
    return np.concatenate([[0], np.sort(mid), [M - 1]])


def run_oracle(prob, rows=None):
    x1 = prob.x1.reshape(-1, prob.K)
    res = prob.residual.reshape(-1, prob.N)
    if rows is not None:
        idx = torch.as_tensor(rows, device=x1.device)
        x1 = x1.index_select(0, idx)
        res = res.index_select(0, idx)
    q = prob.x2.to("cpu").to(torch.int32)
    return oracle.matmul_add_rmsnorm(x1.cpu(), q, prob.scale.cpu(),
                                     None if prob.offset is None else prob.offset.cpu(),
                                     None if prob.bias is None else prob.bias.cpu(), res.cpu(),
                                     prob.gamma.cpu(), prob.eps, prob.group)


def compare(prob, y, no, ref, rows=None, tol=None):
    tol = TOL[prob.dtype] if tol is None else tol
    _, ry, rn = ref
    yg = y.reshape(-1, prob.N)
    ng = no.reshape(-1, prob.N)
    if rows is not None:
        idx = torch.as_tensor(rows, device=yg.device)
        yg = yg.index_select(0, idx)
        ng = ng.index_select(0, idx)
    yg = yg.double().cpu().numpy()
    ng = ng.double().cpu().numpy()
    out = {}
    for name, g, r in (("y", yg, ry), ("normOut", ng, rn)):
        err = np.abs(g - r) / (1.0 + np.abs(r))
        out[name] = float(err.max()) if err.size else 0.0
        bad = np.argwhere(~(err <= tol))
        assert bad.size == 0, (f"{prob.name} {name}: {len(bad)} elements exceed tol {tol}; "
                               f"worst {out[name]:.3e} at {tuple(bad[0])}: gpu {g[tuple(bad[0])]} "
                               f"ref {r[tuple(bad[0])]}")
    return out


def compare_nonfinite(prob, y, no, ref, tol=None):
    """Comparison for inputs that hold NaN or Inf (IEEE propagation). Where the
    oracle's value is finite the GPU's must be finite and within the tolerance;
    where the oracle's is NaN the GPU's must be NaN; where it is +-Inf the GPU's
    must be the same infinity or NaN (the kernels add the dequantized weight's
    terms in an exact but different order, which can turn an Inf into NaN)."""
    tol = TOL[prob.dtype] if tol is None else tol
    _, ry, rn = ref
    for name, g, r in (("y", y, ry), ("normOut", no, rn)):
        g = g.reshape(-1, prob.N).double().cpu().numpy()
        fin_r, fin_g = np.isfinite(r), np.isfinite(g)
        bad = np.argwhere(fin_r != fin_g)
        assert bad.size == 0, (f"{prob.name} {name}: finiteness differs at {tuple(bad[0])}: gpu "
                               f"{g[tuple(bad[0])]} ref {r[tuple(bad[0])]}")
        assert np.isnan(g[np.isnan(r)]).all(), f"{prob.name} {name}: a NaN of the oracle is not NaN"
        inf = np.isinf(r)
        assert (np.isnan(g[inf]) | (g[inf] == r[inf])).all(), f"{prob.name} {name}: Inf differs"
        err = np.abs(g[fin_r] - r[fin_r]) / (1.0 + np.abs(r[fin_r]))
        assert err.size == 0 or err.max() <= tol, f"{prob.name} {name}: worst {err.max():.3e}"
