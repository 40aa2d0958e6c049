"""Upload a workload's arrays to torch tensors (no arithmetic, storage only)."""
from __future__ import annotations

import numpy as np
import torch


def tensor_of(a: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Storage array -> torch tensor with the same bits (bf16 bits -> bfloat16)."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device)


def upload(wl, device="cuda"):
    """Dict of device tensors: k, v, q [steps][B][Hq][d], seq_lens, block_table, budget."""
    return dict(
        k=tensor_of(wl.K, wl.dtype, device),
        v=tensor_of(wl.V, wl.dtype, device),
        q=tensor_of(wl.q, wl.dtype, device),
        seq_lens=torch.from_numpy(wl.seq_lens.astype(np.int32)).to(device),
        block_table=None if wl.block_table is None
        else torch.from_numpy(wl.block_table.astype(np.int32)).to(device),
        budget=torch.from_numpy(wl.budget.astype(np.int32)).to(device),
    )
