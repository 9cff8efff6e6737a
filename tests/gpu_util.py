"""Helpers for the GPU parity tests: device buffers with guard bands, and
conversions between torch tensors and the oracle's numpy arrays."""
import numpy as np
import torch

GUARD = 64  # elements of canary before and after every receive buffer
CANARY_F32 = 0x7FC01234
CANARY_BF16 = 0x7FAB


def torch_dtype(dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def to_device(x_np, dtype):
    """numpy [N, count] (float32 or bf16 bits) -> list of N device tensors (16-byte aligned rows)."""
    n, count = x_np.shape
    stride = -(-count // 64) * 64 + 2 * GUARD
    if dtype == "f32":
        big = torch.empty((n, stride), dtype=torch.float32, device="cuda")
        big[:, GUARD:GUARD + count] = torch.from_numpy(np.ascontiguousarray(x_np)).cuda()
    else:
        big = torch.empty((n, stride), dtype=torch.int16, device="cuda")
        big[:, GUARD:GUARD + count] = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda()
        big = big.view(torch.bfloat16)
    return big, [big[r, GUARD:GUARD + count] for r in range(n)]


def guarded_outputs(n, count, dtype):
    stride = -(-count // 64) * 64 + 2 * GUARD
    big = torch.empty((n, stride), dtype=torch.int32 if dtype == "f32" else torch.int16, device="cuda")
    big.fill_(CANARY_F32 if dtype == "f32" else CANARY_BF16)
    if dtype == "f32":
        big = big.view(torch.float32)
    else:
        big = big.view(torch.bfloat16)
    return big, [big[r, GUARD:GUARD + count] for r in range(n)]


def check_guards(big, count, dtype):
    raw = big.view(torch.int32 if dtype == "f32" else torch.int16)
    canary = CANARY_F32 if dtype == "f32" else CANARY_BF16
    stride = raw.shape[1]
    lo = raw[:, :GUARD]
    hi = raw[:, GUARD + count:]
    assert bool((lo == canary).all()), "guard band before a receive buffer was written"
    assert bool((hi == canary).all()), "guard band after a receive buffer was written"
    assert hi.shape[1] == stride - GUARD - count


def to_numpy(t, dtype):
    t = t.detach().cpu()
    if dtype == "f32":
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def device_rows_numpy(tensors, dtype):
    return np.stack([to_numpy(t, dtype) for t in tensors])
