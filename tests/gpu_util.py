"""Helpers for the GPU parity tests: allocation, host copies, tolerances."""
import os

import numpy as np
import torch

from structured_sparse_gemm_nm_gb300 import binding as nb

DEV = torch.device("cuda")
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8}
ESIZE = {"f16": 2, "bf16": 2, "i8": 1}


def ensure_lib():
    if not os.path.exists(nb.LIB_PATH):
        from structured_sparse_gemm_nm_gb300.build import build

        build()
    nb.lib()


def dev_bytes(nbytes: int, fill=None) -> torch.Tensor:
    """Device buffer of nbytes (rounded up to 16), optionally filled with a byte value (canary)."""
    t = torch.empty(max(16, (nbytes + 15) // 16 * 16), dtype=torch.uint8, device=DEV)
    if fill is not None:
        t.fill_(fill)
    return t


def bits_of(t: torch.Tensor, dtype: str, shape=None) -> np.ndarray:
    """Host numpy copy of a device buffer as uint16 bit patterns (f16/bf16) or int8."""
    a = t.detach().contiguous().cpu().view(torch.uint8).numpy()
    a = a.view(np.uint16) if ESIZE[dtype] == 2 else a.view(np.int8)
    if shape is not None:
        n = int(np.prod(shape))
        a = a[:n].reshape(shape)
    return a


def u16(t: torch.Tensor, count: int) -> np.ndarray:
    return t.detach().cpu().view(torch.uint8).numpy().view(np.uint16)[:count]


def u32(t: torch.Tensor, count: int) -> np.ndarray:
    return t.detach().cpu().view(torch.uint8).numpy().view(np.uint32)[:count]


def to_dev_bits(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Device tensor of the given bit patterns (uint16 for f16/bf16, int8 for i8)."""
    if dtype == "i8":
        return torch.from_numpy(np.ascontiguousarray(a.astype(np.int8))).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(a.astype(np.uint16)).view(np.int16)).view(TORCH_DT[dtype]).to(DEV)


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """FP16/BF16 product tolerance: max|D - D_ref| <= 1e-2 (|D_ref| + 1) and ||D - D_ref||_F <= 2e-3 ||D_ref||_F."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = 1e-2 * (np.abs(ref) + 1.0)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{what}: {len(bad)} elements out of tolerance, first {bad[:3].tolist()}, max err {err.max()}"
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(got - ref) / nref
        assert rel <= 2e-3, f"{what}: relative Frobenius error {rel}"
