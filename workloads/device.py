"""Upload a workloads.Problem to the GPU with torch (device memory only) and
call the library through its C ABI.  Used by the GPU tests and the benchmark;
holds no attention arithmetic."""
import numpy as np
import torch

from . import synth as W
import shared_prefix_kv_gb300 as ps


def shape_of(p):
    return ps.make_shape(p.num_req, p.num_groups, p.num_q_heads, p.num_kv_heads, p.head_dim,
                         p.block_size, p.max_blocks_per_req, p.num_pool_blocks, p.dtype, p.scale)


def _dev_values(a, dtype):
    if dtype == W.F32:
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


class DeviceProblem:
    def __init__(self, p):
        self.p = p
        self.q = _dev_values(p.q, p.dtype)
        self.pool = _dev_values(p.pool, p.dtype)
        self.bt = torch.from_numpy(np.ascontiguousarray(p.block_table)).cuda()
        self.gor = torch.from_numpy(np.ascontiguousarray(p.group_of_req)).cuda()
        self.plen = torch.from_numpy(np.ascontiguousarray(p.prefix_len)).cuda()
        self.slen = torch.from_numpy(np.ascontiguousarray(p.suffix_len)).cuda()
        self.out = torch.full_like(self.q, float("nan"))
        self.lse = torch.full((p.num_req, p.num_q_heads), float("nan"), device="cuda")

    def plan(self, flags=0):
        # leaf_len: ragged leaf levels, set on problems built by a ragged expansion
        p = self.p
        return ps.Plan(shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len,
                       p.suffix_len, flags=flags, leaf_len=getattr(p, "leaf_len", None))

    def decode(self, plan, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        plan.decode(self.q, self.pool, self.bt, self.gor, self.plen, self.slen, self.out,
                    self.lse, stream=s.cuda_stream)

    def result(self):
        torch.cuda.synchronize()
        return self.out.float().cpu().numpy().astype(np.float64), self.lse.cpu().numpy().astype(np.float64)


def tolerances(p):
    """Parity bounds: max abs error 1e-4 for fp32 inputs, 1e-2 for
    bf16 inputs (outputs are rounded to bf16), 1e-3 for the LSE."""
    return (1e-4, 1e-4) if p.dtype == W.F32 else (1e-2, 1e-3)
