"""Put a synthetic workload (workloads.Workload) on the GPU through the library.

Allocates the device tensors of one step with PyTorch, poisons the pools with
quiet-NaN patterns, and writes the history rows into the pools with the
library's own pa_append_kv.  Used by the GPU tests, smoke() and bench.py;
holds no attention arithmetic and never touches the CPU oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import paged_kv_continuous_pa_gb300 as pa
import workloads as W

TORCH_OF = {W.F32: torch.float32, W.BF16: torch.bfloat16, W.E4M3: torch.uint8}


def to_torch(x: np.ndarray, dtype: int, device="cuda") -> torch.Tensor:
    """numpy f32 / bf16-bits / e4m3-codes array -> tensor of the matching torch dtype."""
    if dtype == W.F32:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    elif dtype == W.BF16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8))
    return t.to(device, non_blocking=False)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def poisoned_pool(wl: W.Workload, device="cuda") -> torch.Tensor:
    shape = wl.pool_shape()
    if wl.kv_dtype == W.F32:
        return torch.full(shape, float("nan"), dtype=torch.float32, device=device)
    if wl.kv_dtype == W.BF16:
        return torch.full(shape, W.POISON[W.BF16], dtype=torch.int16, device=device).view(torch.bfloat16)
    return torch.full(shape, W.POISON[W.E4M3], dtype=torch.uint8, device=device)


@dataclass
class DeviceStep:
    wl: W.Workload
    pool: pa.Pool
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_tables: torch.Tensor
    seq_ids: torch.Tensor
    positions: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    out: torch.Tensor
    workspace: torch.Tensor | None
    status: torch.Tensor

    def append_step(self, stream=None):
        pa.append_kv(self.pool, self.k_new, self.v_new, self.seq_ids, self.positions, self.block_tables,
                     status=self.status, stream=stream)

    def step(self, stream=None, out=None):
        """append_step() and attend() as one pa_step call."""
        pa.step(self.pool, self.q, self.k_new, self.v_new, self.seq_ids, self.positions, self.block_tables,
                self.out if out is None else out, chunks=self.wl.chunks, softmax_scale=self.wl.softmax_scale,
                workspace=self.workspace, status=self.status, stream=stream)

    def attend(self, stream=None, out=None):
        pa.attention(self.pool, self.q, self.seq_ids, self.positions, self.block_tables,
                     self.out if out is None else out, chunks=self.wl.chunks, softmax_scale=self.wl.softmax_scale,
                     workspace=self.workspace, status=self.status, stream=stream)


def upload(wl: W.Workload, device="cuda", hist_batch_rows: int = 1 << 19) -> DeviceStep:
    """Allocate, poison, and fill the pools with the workload's history rows."""
    k_pool, v_pool = poisoned_pool(wl, device), poisoned_pool(wl, device)
    pool = pa.Pool(k_pool, v_pool, wl.k_scale, wl.v_scale)
    bt = torch.from_numpy(wl.block_tables).to(device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for b in range(0, len(wl.hist_seq), hist_batch_rows):
        e = min(len(wl.hist_seq), b + hist_batch_rows)
        pa.append_kv(pool, to_torch(wl.hist_k[b:e], wl.in_dtype, device), to_torch(wl.hist_v[b:e], wl.in_dtype, device),
                     torch.from_numpy(wl.hist_seq[b:e]).to(device), torch.from_numpy(wl.hist_pos[b:e]).to(device),
                     bt, status=status)
    q = to_torch(wl.q, wl.q_dtype, device)
    ws_bytes = pa.workspace_bytes(pool, wl.n_rows, wl.Hq, wl.max_blocks, wl.chunks)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device) if ws_bytes else None
    step = DeviceStep(wl=wl, pool=pool, k_pool=k_pool, v_pool=v_pool, block_tables=bt,
                      seq_ids=torch.from_numpy(wl.seq_ids).to(device),
                      positions=torch.from_numpy(wl.positions).to(device), q=q,
                      k_new=to_torch(wl.k_new, wl.in_dtype, device), v_new=to_torch(wl.v_new, wl.in_dtype, device),
                      out=torch.empty_like(q), workspace=ws, status=status)
    torch.cuda.synchronize()
    return step
