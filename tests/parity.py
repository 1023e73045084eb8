"""Comparison helpers shared by the GPU parity tests.

Tolerances (the codec's stated parity bar):
  * FP8 codes: at least 99.99 % bit-identical, never more than 1 E4M3 ULP
    apart (codes compared as sign-magnitude integers, +0 == -0);
  * per-block fp32 scalars alpha and s: within 1e-6 relative;
  * reconstructions, judged on the same codes: relative L2 error per tensor
    and max error per block (relative to the block's max) within 1e-6.
"""

from __future__ import annotations

import numpy as np
import torch

CODE_MATCH = 0.9999
SCALAR_RTOL = 1e-6
RECON_RTOL = 1e-6

# Statistics of the comparisons made during a test session, written out as
# JSON at the end when TACO_PARITY_REPORT names a file (see conftest.py).
REPORT: dict = {}
_CURRENT = {"test": "?"}


def _record(kind: str, what: str, value) -> None:
    entry = REPORT.setdefault(_CURRENT["test"], {})
    key = f"{kind}:{what}"
    old = entry.get(key)
    if isinstance(value, dict):
        if old is None:
            entry[key] = dict(value)
        else:
            old["identical"] = min(old["identical"], value["identical"])
            old["max_ulp"] = max(old["max_ulp"], value["max_ulp"])
    else:
        entry[key] = value if old is None else max(old, value)


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = a.astype(np.int32).reshape(-1)
    b = b.astype(np.int32).reshape(-1)
    ma, mb = a & 0x7F, b & 0x7F
    sa = np.where(ma == 0, 1, np.where(a >> 7, -1, 1))
    sb = np.where(mb == 0, 1, np.where(b >> 7, -1, 1))
    return np.abs(sa * ma - sb * mb)


def assert_codes_match(gpu: np.ndarray, ref: np.ndarray, what: str = "codes", exact: bool = False) -> dict:
    if exact:
        bad = np.flatnonzero(gpu.reshape(-1) != ref.reshape(-1))
        assert bad.size == 0, f"{what}: {bad.size} codes differ, first at {bad[:5]}"
    d = ulp_distance(gpu, ref)
    same = float(np.mean(d == 0))
    worst = int(d.max()) if d.size else 0
    assert not np.any((gpu.reshape(-1) & 0x7F) == 0x7F), f"{what}: NaN code emitted"
    assert same >= CODE_MATCH and worst <= 1, f"{what}: identical {same:.6f}, max ULP {worst}"
    stats = {"identical": same, "max_ulp": worst}
    _record("codes", what, stats)
    return stats


def assert_scalars_match(gpu: np.ndarray, ref: np.ndarray, what: str, rtol: float = SCALAR_RTOL,
                         exact: bool = False) -> float:
    if exact:
        assert np.array_equal(gpu.reshape(-1), ref.reshape(-1)), f"{what}: not bit-identical"
    g = gpu.astype(np.float64).reshape(-1)
    r = ref.astype(np.float64).reshape(-1)
    assert np.all(np.isfinite(g)), f"{what}: non-finite"
    err = np.abs(g - r) / np.where(r == 0, 1.0, np.abs(r))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= rtol, f"{what}: max relative error {worst:.3e} at block {int(err.argmax())}"
    _record("scalar_max_rel", what, worst)
    return worst


def assert_recon_match(gpu: np.ndarray, ref: np.ndarray, block: int, what: str = "recon",
                       rtol: float = RECON_RTOL) -> float:
    g = gpu.astype(np.float64).reshape(-1, block)
    r = ref.astype(np.float64).reshape(-1, block)
    nrm = np.linalg.norm(r)
    rel = float(np.linalg.norm(g - r) / nrm) if nrm > 0 else float(np.linalg.norm(g))
    assert rel <= rtol, f"{what}: relative L2 {rel:.3e}"
    bmax = np.abs(r).max(axis=1)
    berr = np.abs(g - r).max(axis=1)
    assert np.all(berr <= rtol * bmax), f"{what}: block max error {float((berr / np.where(bmax == 0, 1, bmax)).max()):.3e}"
    _record("recon_rel_l2", what, rel)
    return rel


def sample_blocks(nb: int, k: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = rng.choice(nb, size=min(k, nb), replace=False)
    return np.unique(np.concatenate([pick, [0, nb - 1]]))


def gather_blocks(t: torch.Tensor, blocks: np.ndarray, block: int) -> np.ndarray:
    """Rows of a [nb, block] view of a device tensor, copied to the host."""
    idx = torch.from_numpy(blocks).to(t.device)
    return to_host(t.reshape(-1, block).index_select(0, idx))


def gather_scalars(t: torch.Tensor, blocks: np.ndarray) -> np.ndarray:
    idx = torch.from_numpy(blocks).to(t.device)
    return to_host(t.reshape(-1).index_select(0, idx))
