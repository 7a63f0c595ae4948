"""Shared helpers for the GPU parity tests: run the CUDA path, compare with the oracle.

Tolerances (on the bf16 output, against the binary64 oracle):
  * max |gpu - oracle| <= 8e-3 and mean |gpu - oracle| <= 2e-4 per batch,
    literally, on the benchmark-shaped batches (the workloads the bar is
    quoted on: long contexts, so |o| is an average of many values);
  * an element whose exact value has |o| >= 4 has a bf16 spacing of 2^-5 or
    more: rounding the exact value alone can cost 2^-6 = 0.0156, more than
    the 8e-3 bar, so its bound is 8e-3 plus half a bf16 step at |o|; such
    elements are counted and reported. Below 4 the bar is literal: in
    [2, 4) the nearest bf16 is at most 2^-7 = 0.0078 away, which leaves the
    kernel 1.9e-4 of its own error near a rounding midpoint;
  * on edge-case batches with a few tokens, |o| is O(1) and rounding the
    exact value to bf16 alone costs about |o|/1000 on average, more than
    2e-4; there the mean bar is 2e-4 on top of that unavoidable rounding
    error (mean |bf16(oracle) - oracle|), which is computed and reported.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_decode_pda_gb300 as pda

MAX_ABS = 8e-3
MEAN_ABS = 2e-4
# |o| from which bf16 itself cannot meet MAX_ABS (half its spacing exceeds it)
BF16_LIMITED = 4.0


def run_cuda(batch, out=None, stream=None) -> torch.Tensor:
    cfg = batch.cfg
    return pda.decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                      cfg.k_scale, cfg.v_scale, out=out, stream=stream)


def run_oracle(batch, seq_ids=None) -> np.ndarray:
    cfg = batch.cfg
    return oracle.decode(**batch.raw(), scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale,
                         seq_ids=seq_ids)


def bf16_half_step(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers around |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def compare(got_bf16: torch.Tensor, ref: np.ndarray, label: str = "", literal: bool = False) -> dict:
    got = got_bf16.detach().float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "%s: non-finite output" % label
    err = np.abs(got - ref)
    big = np.abs(ref) >= BF16_LIMITED
    bound = np.where(big, MAX_ABS + bf16_half_step(ref), MAX_ABS)
    worst = float(err.max()) if err.size else 0.0
    mean = float(err.mean()) if err.size else 0.0
    # error beyond the unavoidable bf16 rounding of the exact value
    rounded = ref.astype(np.float32)
    rounded = torch.from_numpy(rounded).to(torch.bfloat16).float().numpy().astype(np.float64)
    repr_err = float(np.abs(rounded - ref).mean()) if ref.size else 0.0
    stats = dict(max_abs=worst, mean_abs=mean, max_abs_vs_bf16_oracle=float(np.abs(got - rounded).max()),
                 mean_abs_bf16_rounding_of_oracle=repr_err,
                 max_abs_out=float(np.abs(ref).max()) if ref.size else 0.0, n_bf16_limited=int(big.sum()),
                 n_out_2_to_4=int(((np.abs(ref) >= 2.0) & ~big).sum()))
    if not (err <= bound).all():
        at = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: max abs err %g (bound %g) at %s: gpu %r oracle %r" % (
            label, worst, float(bound[at]), at, float(got[at]), float(ref[at])))
    mean_bar = MEAN_ABS if literal else MEAN_ABS + repr_err
    assert mean <= mean_bar, "%s: mean abs err %g > %g (bf16 rounding of the exact value alone: %g)" % (
        label, mean, mean_bar, repr_err)
    return stats


def compare_e4m3(got_u8: torch.Tensor, exact: np.ndarray, out_scale: float, label: str = "",
                 min_equal: float = 0.9) -> dict:
    """Check an e4m3 output (codes of o / out_scale) against the exact result.

    The kernel decides each code on its fp32 result, the oracle on the exact
    one. Per element the stored value lies within half an e4m3 step at |o|
    (the rounding any e4m3 output has) plus the 8e-3 bar of the bf16 path;
    values past 448 * out_scale saturate to +-448 on both sides. On average
    the kernel adds at most the 2e-4 mean bar to the e4m3 rounding error of
    the exact values, and most codes equal the code of the exact result.
    """
    got = got_u8.view(torch.uint8).cpu().numpy()
    want = oracle.quantize_e4m3(exact, out_scale)
    vg = torch.from_numpy(got).view(torch.float8_e4m3fn).double().numpy() * out_scale
    vw = torch.from_numpy(want).view(torch.float8_e4m3fn).double().numpy() * out_scale
    target = np.clip(exact, -448.0 * out_scale, 448.0 * out_scale)
    q = np.abs(target) / out_scale
    expo = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    half_step = np.ldexp(1.0, (expo - 4).astype(np.int64)) * out_scale
    err = np.abs(vg - target)
    assert np.isfinite(vg).all(), "%s: non-finite e4m3 code" % label
    assert np.all(err <= half_step + MAX_ABS), "%s: max excess %g" % (label, float(np.max(err - half_step)))
    mean_w = float(np.abs(vw - target).mean()) if err.size else 0.0
    assert err.mean() <= mean_w + MEAN_ABS, "%s: mean %g vs exact-code mean %g" % (label, err.mean(), mean_w)
    frac_equal = float(np.mean(got == want)) if err.size else 1.0
    assert frac_equal >= min_equal, "%s: only %.4f of e4m3 codes equal the exact result's code" % (
        label, frac_equal)
    return dict(frac_equal=frac_equal, mean=float(err.mean()) if err.size else 0.0)
