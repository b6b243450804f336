"""Helpers for the GPU tests: move seeded canonical inputs to the device, pack them with the
library, and compare bf16 outputs with the fp64 oracle."""
import numpy as np
import torch

TOL = 5e-3  # max|y - y_ref| / max|y_ref|


def dev_u32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).cuda()


def dev_u16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda()


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return dev_u16(a).view(torch.bfloat16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def pack_q4(nq, wq: np.ndarray, s: np.ndarray, K: int, N: int):
    """Packed weight (one uint8 device tensor)."""
    return nq.pack_q4(dev_u32(wq), dev_u16(s), K, N)


def pack_q5(nq, wn: np.ndarray, wh: np.ndarray, s: np.ndarray, K: int, N: int):
    return nq.pack_q5(dev_u32(wn), dev_u32(wh), dev_u16(s), K, N)


def rel_err(y: np.ndarray, y_ref: np.ndarray) -> float:
    m = float(np.max(np.abs(y_ref)))
    return float(np.max(np.abs(y - y_ref))) / (m if m > 0 else 1.0)


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """First and last rows, both halves of a 16-row tile, plus random rows."""
    g = np.random.default_rng(seed)
    fixed = [0, 7, 8, 15, 16, N // 2, N - 17, N - 16, N - 9, N - 1]
    rnd = g.choice(N, size=min(count, N), replace=False)
    return np.unique(np.clip(np.concatenate([fixed, rnd]), 0, N - 1)).astype(np.int32)


def expect_timeout(nq, call, tries=5):
    """Run `call` with a 1 ns wait bound until nq_device_error reports a timeout (a block
    whose every wait is satisfied at the first look cannot time out, so allow a few tries)."""
    import pytest
    from weight_only_groupwise_gb300.nq import NqError
    for _ in range(tries):
        prev = nq.wait_limit(1)
        try:
            call()
        finally:
            nq.wait_limit(prev)
        try:
            nq.device_error()
        except NqError as e:
            assert e.status == -7, e
            nq.device_error()          # reported once, then clear
            return
    pytest.fail("no bounded wait ran out with a 1 ns bound")
