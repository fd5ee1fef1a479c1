"""Helpers of the GPU parity tests: inputs as torch tensors, the oracle over
row chunks (for full-size batches), and the comparison rules.

Tolerances (fp32 arithmetic on the GPU against the fp64 oracle):
  * bit-exact: idx, counts, rank_load, perm, slot, offsets, kept, n_dropped
  * gate, f, P, scalars:  |x - o| <= 1e-5 * |o|
  * dlogits:              |x - o| <= 1e-5 * (|o| + c * p_tj * (|f_j| + |s_t|)),
                          c = grad_scale * alpha * E / T, s_t = sum_i p_ti f_i: the gradient
                          c * p_tj * (f_j - s_t) is a difference that cancels, so 1e-5
                          relative is taken against the magnitude of its two terms
  * Sinkhorn u, v, plan:  |x - o| <= 1e-4 * |o| + 1e-4 * max|o| per microbatch
  * every floating comparison of the router outputs also admits an absolute
    error of FLT_MIN = 2^-126: fp32 results below the smallest normal number
    carry no relative precision, and the kernels' exponentials flush them to
    zero (a row whose logits spread by more than about 87 gives such p)
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

RTOL = 1e-5
SK_RTOL = 1e-4
FLT_MIN = 2.0 ** -126
SCALARS = ("l_aux", "balance", "cv", "max_over_mean", "min_over_mean", "rank_cv", "rank_max_over_mean")


def to_device(logits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(logits).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(device)


def assert_close(name: str, got, want, rtol: float, atol: float = 0.0) -> None:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    err = np.abs(got - want)
    bound = rtol * np.abs(want) + atol
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r} (|err| {err[i]:.3e} > {bound[i]:.3e})")


def assert_equal(name: str, got, want) -> None:
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if not np.array_equal(got.astype(np.int64), want.astype(np.int64)):
        diff = np.argwhere(got.astype(np.int64) != want.astype(np.int64))
        raise AssertionError(f"{name}: {len(diff)} mismatches, first at {diff[0].tolist()}: "
                             f"got {got[tuple(diff[0])]} want {want[tuple(diff[0])]}")


def oracle_forward(logits: np.ndarray, dtype: str, k: int, alpha: float, renorm: bool | None,
                   n_ranks: int, chunk: int = 16384) -> dict:
    """The oracle's router forward, taken over row chunks (row-wise steps per
    chunk; counts and P over the whole batch)."""
    T, E = logits.shape
    if renorm is None:
        renorm = k > 1
    idx = np.empty((T, k), dtype=np.int64)
    gate = np.empty((T, k))
    psum = np.zeros(E)
    for r0 in range(0, T, chunk):
        z = oracle.router.widen(logits[r0:r0 + chunk], dtype)
        p = oracle.router.softmax(z)
        i = oracle.router.top_k(z, k)
        idx[r0:r0 + chunk] = i
        gate[r0:r0 + chunk] = oracle.router.gates(p, i, renorm)
        psum += oracle.router.mean_router_prob(p) * z.shape[0]
    out = oracle.router.batch_statistics(oracle.router.expert_counts(idx, E), psum / T, T, k, alpha, n_ranks)
    out["idx"], out["gate"] = idx, gate
    return out


def check_forward(got: dict, want: dict, n_ranks: int) -> None:
    assert_equal("idx", got["idx"].cpu().numpy(), want["idx"])
    assert_close("gate", got["gate"].cpu().numpy(), want["gate"], RTOL, FLT_MIN)
    assert_equal("counts", got["counts"].cpu().numpy(), want["counts"])
    assert_close("f", got["f"].cpu().numpy(), want["f"], RTOL)
    assert_close("P", got["P"].cpu().numpy(), want["P"], RTOL, FLT_MIN)
    sc = got["scalars"].cpu().numpy()
    for j, name in enumerate(SCALARS):
        assert_close(f"scalar {name}", sc[j], want[name], RTOL)
    if n_ranks > 0:
        assert_equal("rank_load", got["rank_load"].cpu().numpy(), want["rank_load"])


def check_backward(dlogits: torch.Tensor, logits: np.ndarray, dtype: str, f: np.ndarray, alpha: float,
                   grad_scale: float, chunk: int = 16384) -> None:
    T, E = logits.shape
    got = dlogits.cpu().numpy()
    c = grad_scale * alpha * E / T
    for r0 in range(0, T, chunk):
        sl = logits[r0:r0 + chunk]
        want = oracle.router.aux_loss_grad(sl, dtype, f, alpha, grad_scale, T=T)
        p = oracle.router.softmax(oracle.router.widen(sl, dtype))
        s = (p * f[None, :]).sum(axis=1)
        scale = abs(c) * p * (np.abs(f)[None, :] + np.abs(s)[:, None])
        assert_close(f"dlogits rows {r0}..", got[r0:r0 + chunk], want, RTOL, RTOL * scale + FLT_MIN)


def check_dispatch(got: dict, idx: np.ndarray, E: int, C: int) -> None:
    want = oracle.dispatch.dispatch(idx, E, C)
    assert_equal("perm", got["perm"].cpu().numpy(), want["perm"])
    assert_equal("slot", got["slot"].cpu().numpy(), want["slot"])
    assert_equal("offsets", got["offsets"].cpu().numpy(), want["offsets"])
    assert_equal("kept", got["kept"].cpu().numpy(), want["kept"])
    assert_equal("n_dropped", got["n_dropped"].cpu().numpy()[0], want["n_dropped"])


def workload_inputs(name: str, T: int | None = None):
    w = synth.ROUTER_WORKLOADS[name]
    if T is not None and T != w.T:
        w = w.with_tokens(T)
    return w, synth.router_logits(w)
