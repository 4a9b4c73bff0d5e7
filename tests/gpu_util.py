"""Helpers for the GPU tests: move a workloads.Problem to the device, run it
through the C ABI, bring D back as bf16 bit patterns."""
from __future__ import annotations

import numpy as np

SENTINEL = 0x7FA5          # a bf16 NaN payload no GEMM result can produce


def dev_tensors(p, device="cuda"):
    import torch
    t = {
        "A": torch.from_numpy(np.ascontiguousarray(p.A)).to(device),
        "SFA": torch.from_numpy(np.ascontiguousarray(p.SFA)).to(device),
        "B": torch.from_numpy(np.ascontiguousarray(p.B)).to(device),
        "SFB": torch.from_numpy(np.ascontiguousarray(p.SFB)).to(device),
    }
    if p.m_indices is not None:
        t["layout"] = torch.from_numpy(np.ascontiguousarray(p.m_indices, dtype=np.int32)).to(device)
    if p.masked_m is not None:
        t["layout"] = torch.from_numpy(np.ascontiguousarray(p.masked_m, dtype=np.int32)).to(device)
    if p.C is not None:
        t["C"] = torch.from_numpy(np.ascontiguousarray(p.C, dtype=np.float32)).to(device)
    return t


def new_d(p, device="cuda", fill=SENTINEL):
    import torch
    D = torch.empty(p.d_shape(), dtype=torch.bfloat16, device=device)
    D.view(torch.int16).fill_(np.int16(np.uint16(fill).view(np.int16)))
    return D


def call(p, t, D, workspace=None, stream=None, layout=None) -> int:
    import fp8_block_scaled_persistent_gb300 as fg
    if p.kind == "nt":
        return fg.fp8_gemm_nt(t["A"], t["SFA"], t["B"], t["SFB"], D, p.M, p.N, p.K,
                              workspace=workspace, stream=stream)
    if p.kind == "nt_ue8m0":
        return fg.fp8_gemm_nt_ue8m0(t["A"], t["SFA"], t["B"], t["SFB"], D, p.M, p.N, p.K, stream=stream)
    if p.kind == "nt_acc":
        return fg.fp8_gemm_nt_accumulate(t["A"], t["SFA"], t["B"], t["SFB"], t["C"], D, p.M, p.N, p.K,
                                         workspace=workspace, stream=stream)
    lay = t["layout"] if layout is None else layout
    if p.kind == "contiguous":
        return fg.fp8_gemm_grouped_contiguous(t["A"], t["SFA"], t["B"], t["SFB"], D, lay,
                                              p.M, p.N, p.K, p.G, workspace=workspace, stream=stream)
    return fg.fp8_gemm_grouped_masked(t["A"], t["SFA"], t["B"], t["SFB"], D, lay,
                                      p.G, p.M, p.N, p.K, workspace=workspace, stream=stream)


def bits(D) -> np.ndarray:
    import torch
    torch.cuda.synchronize()
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def workspace_for(p, device="cuda"):
    """A zero-filled workspace of the size the library asks for (None if 0)."""
    import torch
    import fp8_block_scaled_persistent_gb300 as fg
    if p.kind == "nt_ue8m0":
        return None
    kind = {"nt": 0, "nt_acc": 0, "contiguous": 1, "masked": 2}[p.kind]
    n = fg.fp8_gemm_workspace_size(kind, p.M, p.N, p.K, p.G)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def run(p, workspace="auto", D=None):
    """Runs p through the C ABI; returns (D bits, status, device status)."""
    import fp8_block_scaled_persistent_gb300 as fg
    t = dev_tensors(p)
    if D is None:
        D = new_d(p)
    ws = workspace_for(p) if workspace == "auto" else workspace
    st = call(p, t, D, workspace=ws)
    dst = fg.fp8_gemm_get_device_error()
    return bits(D), st, dst


def sample_rows(M, count, seed=0, must=()):
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in must if 0 <= r < M)
    rows.update(int(r) for r in rng.choice(M, size=min(count, M), replace=False))
    return np.array(sorted(rows), dtype=np.int32)
