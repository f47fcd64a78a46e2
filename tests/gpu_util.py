"""Helpers for the GPU parity tests: upload seeded inputs, run the library through
its binding, compare with the oracle under the stated tolerance."""

from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np
import pytest
import torch

import oracle

from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W

# Tolerances of the path (bf16 in, fp32 accumulate): max |err| <= 2e-2 and relative L2
# <= 5e-3 against the fp64 oracle.  A bf16 output cannot be closer to the exact value
# than half a bf16 ulp, so the per-element bound adds half an ulp of the oracle value.
MAX_ABS = 2e-2
MAX_REL_L2 = 5e-3


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def to_dev_bits(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits -> device bf16 tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def ids_dev(ids: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()


def bf16_half_ulp(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * np.exp2(e - 7)


def compare_bf16(y_gpu_bits: np.ndarray, y_ref: np.ndarray, what: str = ""):
    """Assert the bf16 GPU output matches the fp64 oracle; return (max_abs, rel_l2)."""
    g = W.bf16_bits_to_f32(y_gpu_bits).astype(np.float64)
    assert g.shape == y_ref.shape
    assert np.isfinite(g).all(), what + ": non-finite output"
    err = np.abs(g - y_ref)
    bound = MAX_ABS + bf16_half_ulp(y_ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    assert (err <= bound).all(), "%s: |err| %.4g > bound %.4g at %s" % (
        what, err[worst], bound[worst], worst)
    denom = np.linalg.norm(y_ref)
    rel = float(np.linalg.norm(g - y_ref) / denom) if denom > 0 else 0.0
    assert rel <= MAX_REL_L2, "%s: rel L2 %.3g" % (what, rel)
    return float(err.max(initial=0.0)), rel


def new_err() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_apply(batch: W.Batch, pool_host: W.AdapterPool, mode: int, n_adapters: int, view=None,
              ids=None):
    """Segments + fused apply on the GPU; returns (y bits [T, ldy], err word, segments)."""
    view = view or B.PoolView.from_host(pool_host)
    ids = batch.ids if ids is None else ids
    x = to_dev_bits(batch.x)
    y = to_dev_bits(batch.y0)
    idt = ids_dev(ids)
    seg = B.Segments(len(ids))
    err = new_err()
    B.lora_segments_build(idt, n_adapters, seg, mode=mode, err=err)
    B.lora_apply(x, y, seg, view, err=err)
    torch.cuda.synchronize()
    return to_host_bits(y), int(err.item()), seg


def run_bgmv(batch: W.Batch, pool_host: W.AdapterPool, view=None, ids=None):
    view = view or B.PoolView.from_host(pool_host)
    ids = batch.ids if ids is None else ids
    x = to_dev_bits(batch.x)
    y = to_dev_bits(batch.y0)
    err = new_err()
    B.lora_bgmv(x, y, ids_dev(ids), view, err=err)
    torch.cuda.synchronize()
    return to_host_bits(y), int(err.item())


def compare_f32(yf: np.ndarray, y_ref: np.ndarray, what: str = ""):
    """Assert an fp32 GPU output meets the literal bounds against the fp64 oracle:
    max |err| <= 2e-2 and relative L2 <= 5e-3 (no allowance for output rounding, since
    the fp32 output is not rounded to bf16); return (max_abs, rel_l2)."""
    g = np.asarray(yf, dtype=np.float64)
    assert g.shape == y_ref.shape
    assert np.isfinite(g).all(), what + ": non-finite output"
    err = np.abs(g - y_ref)
    mx = float(err.max(initial=0.0))
    assert mx <= MAX_ABS, "%s: max |err| %.4g > %g" % (what, mx, MAX_ABS)
    denom = np.linalg.norm(y_ref)
    rel = float(np.linalg.norm(g - y_ref) / denom) if denom > 0 else 0.0
    assert rel <= MAX_REL_L2, "%s: rel L2 %.3g" % (what, rel)
    return mx, rel


def oracle_apply(x, y0, ids, pool, threads: int = 0):
    """The oracle's y over the given rows, its rows split across host threads (each
    token's result is independent; the C oracle holds no global state and runs
    without the interpreter lock)."""
    n = threads or min(16, os.cpu_count() or 1)
    T = len(ids)
    if T < 64 or n <= 1:
        return oracle.lora_apply(x, y0, ids, pool)
    bounds = np.linspace(0, T, n + 1).astype(int)
    with ThreadPoolExecutor(max_workers=n) as ex:
        parts = list(ex.map(lambda i: oracle.lora_apply(x[bounds[i]:bounds[i + 1]], y0[bounds[i]:bounds[i + 1]],
                                                        ids[bounds[i]:bounds[i + 1]], pool),
                            range(n)))
    err = 0
    for _, e in parts:
        err |= e
    return np.concatenate([y for y, _ in parts], axis=0), err


def run_apply_f32y(batch: W.Batch, pool_host: W.AdapterPool, mode: int, n_adapters: int, view=None):
    """Segments + lora_apply_f32y; returns (yf [T, d_out] fp32, err word).  Rows the call
    does not write keep the NaN they start with."""
    view = view or B.PoolView.from_host(pool_host)
    x = to_dev_bits(batch.x)
    y0 = to_dev_bits(batch.y0)
    yf = torch.full((batch.T, pool_host.d_out), float("nan"), dtype=torch.float32, device="cuda")
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), n_adapters, seg, mode=mode, err=err)
    B.lora_apply_f32y(x, y0, yf, seg, view, err=err)
    torch.cuda.synchronize()
    return yf.cpu().numpy(), int(err.item())
