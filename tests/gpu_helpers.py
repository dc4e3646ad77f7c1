"""Shared checks for the GPU parity tests (comparisons only, no method arithmetic)."""

import numpy as np
import torch

# Output tolerance for bf16 / fp16 inputs with fp32 accumulation, fp32 output.
ATOL = 2e-3
# Selection band: where the oracle's K-th and (K+1)-th scores are closer than
# this (relative), pages whose scores lie within the band may be swapped.
SEL_REL = 1e-5


def require_cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import decode_attention_paged_kv_gb300 as dkv
    dkv.lib()  # raises if the library is missing
    return torch.device("cuda:0")


def check_selection(gpu_sel: np.ndarray, r: np.ndarray, K: int):
    """gpu_sel [rows, kk] ascending page indices vs oracle scores r [rows, P].

    Valid iff: kk distinct, ascending, in range; every page scoring above
    r_K + band is selected; every selected page scores at least r_K - band,
    where r_K is the oracle's K-th largest score and band = 1e-5 * max(|r_K|, 1e-30).
    Returns the number of rows whose set differs from the oracle's exact top-K.
    """
    rows, P = r.shape
    kk = min(K, P)
    assert gpu_sel.shape == (rows, kk)
    swaps = 0
    for i in range(rows):
        s = gpu_sel[i]
        assert np.all(np.diff(s) > 0), f"row {i}: not strictly ascending"
        assert s.min() >= 0 and s.max() < P
        order = sorted(range(P), key=lambda j: (-r[i, j], j))
        rk = r[i, order[kk - 1]]
        band = SEL_REL * max(abs(rk), 1e-30)
        chosen = np.zeros(P, bool)
        chosen[s] = True
        must = r[i] > rk + band
        assert np.all(chosen[must]), f"row {i}: a page above the band was dropped"
        assert np.all(r[i][chosen] >= rk - band), f"row {i}: a page below the band was taken"
        if set(s.tolist()) != set(order[:kk]):
            swaps += 1
    return swaps


def max_abs(a, b) -> float:
    a = a.detach().cpu().double().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)
    b = b.detach().cpu().double().numpy() if isinstance(b, torch.Tensor) else np.asarray(b)
    return float(np.abs(a - b).max())
