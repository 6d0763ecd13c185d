"""Helpers for the GPU parity tests: move seeded numpy inputs to the device, run the
C-ABI path, bring results back as numpy arrays in the oracle's conventions (bf16 as
uint16 bit patterns, e4m3 as uint8)."""
from __future__ import annotations

import numpy as np
import torch

import combine_layout_02_gb300 as ep
from combine_layout_02_gb300.buffers import LayoutBuffers, LLBuffers, RecvBuffers

ATOL, RTOL = 1e-3, 1e-2          # combine tolerance (bf16 output, fp32 accumulation)


def dev_bf16(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def assert_close_bf16(got_bits, exp_bits, atol=ATOL, rtol=RTOL):
    g, e = bf16_to_f64(got_bits), bf16_to_f64(exp_bits)
    bad = np.abs(g - e) > atol + rtol * np.abs(e)
    assert not bad.any(), f"{bad.sum()} elements outside tolerance; first at {np.argwhere(bad)[0]}"


def assert_close_bf16_dev(got: torch.Tensor, exp_bits: np.ndarray, atol=ATOL, rtol=RTOL,
                          chunk=1 << 24):
    """assert_close_bf16 for a device bf16 tensor against expected bf16 bit patterns,
    evaluated on the device in float64 chunk by chunk (full-size outputs)."""
    g_all = got.reshape(-1)
    e_all = np.ascontiguousarray(exp_bits).reshape(-1)
    assert g_all.numel() == e_all.size, (g_all.numel(), e_all.size)
    for i in range(0, e_all.size, chunk):
        e = torch.from_numpy(e_all[i:i + chunk].view(np.int16)).cuda().view(torch.bfloat16).double()
        g = g_all[i:i + chunk].double()
        bad = (g - e).abs() > atol + rtol * e.abs()
        if bool(bad.any()):
            first = i + int(torch.nonzero(bad)[0].item())
            raise AssertionError(f"{int(bad.sum().item())} elements outside tolerance in chunk at "
                                 f"{i}; first at flat index {first}")


U_FP32 = 2.0 ** -24             # unit roundoff of binary32


def assert_weight_sums_close(got, exp, recv_topk_weights, send_head, row_offset):
    """combined_topk_weights against the oracle. The kernel adds each token's received
    weights in fp32, one destination row after another (n terms); the oracle adds them in
    binary64 and rounds once. The recursive-summation bound (Higham, "Accuracy and Stability
    of Numerical Algorithms", 2nd ed., section 4.2) gives, per element,
        |got - exact| <= (n - 1) u sum_i |x_i| / (1 - (n - 1) u),   u = 2^-24,
    and the oracle's rounding adds at most u |exp|; the test allows that plus 1 %."""
    got = np.asarray(got, np.float64)
    exp = np.asarray(exp, np.float64)
    R, T = send_head.shape[0], send_head.shape[1]
    k = recv_topk_weights.shape[1]
    got, exp = got.reshape(R, T, k), exp.reshape(R, T, k)
    sabs = np.zeros((R, T, k))
    n = np.zeros((R, T, 1))
    for d in range(R):
        h = send_head[:, :, d]
        m = h >= 0
        sabs[m] += np.abs(recv_topk_weights[int(row_offset[d]) + h[m]].astype(np.float64))
        n[m] += 1
    g = np.maximum(n - 1, 0) * U_FP32
    tol = (g / (1 - g) * sabs + U_FP32 * np.abs(exp)) * 1.01 + 1e-37
    bad = np.abs(got - exp) > tol
    assert not bad.any(), (f"{int(bad.sum())} weight sums outside the fp32 summation bound; first at "
                           f"{np.argwhere(bad)[0]}: {got[bad][0]} vs {exp[bad][0]}")


def compact_offsets(rank_prefix: np.ndarray) -> list:
    off = [0]
    for n in rank_prefix[-1]:
        off.append(off[-1] + int(n))
    return off


class GpuRun:
    """Holds device inputs and buffers of one workload."""

    def __init__(self, R, T, H, E, k, C, inp, nmax=0):
        self.R, self.T, self.H, self.E, self.k, self.C = R, T, H, E, k, C
        self.sh = ep.make_shape(R, T, H, E, k, C, nmax=nmax)
        self.inp = inp
        self.topk = torch.from_numpy(np.ascontiguousarray(inp["topk_idx"])).cuda()
        self.wts = torch.from_numpy(np.ascontiguousarray(inp["topk_weights"])).cuda()
        self.x = dev_bf16(inp["x"]) if inp.get("x") is not None else None
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.launch = ep.make_launch(error_flags=self.err)
        self.lb = None

    def flags(self) -> int:
        torch.cuda.synchronize()
        return int(self.err.item())

    def layout(self) -> dict:
        self.lb = LayoutBuffers(self.sh)
        ep.ep_get_layout(self.sh, self.topk, self.lb.layout(), self.lb.handle(), self.lb.workspace,
                         self.launch)
        return {k: v.cpu().numpy() for k, v in self.lb.as_dict().items()}

    def dispatch(self, off, recv_dtype=ep.EP_BF16, with_topk=True, x=None, x_dtype=ep.EP_BF16,
                 x_scales=None, fill=0xA5, fp8_scale=ep.EP_FP8_SCALE_FP32,
                 tensor_scale=0.0) -> RecvBuffers:
        rb = RecvBuffers(off[-1], self.H, self.k, recv_dtype=recv_dtype, with_topk=with_topk, fill=fill,
                         fp8_scale=fp8_scale)
        ep.ep_dispatch(self.sh, self.x if x is None else x, x_dtype, x_scales, recv_dtype,
                       self.topk if with_topk else None, self.wts if with_topk else None,
                       self.lb.handle(rb.recv_src_idx), rb.recv_x, rb.recv_x_scales,
                       rb.recv_topk_idx, rb.recv_topk_weights, rb.recv_src_idx, off, self.launch,
                       fp8_scale=fp8_scale, tensor_scale=tensor_scale)
        return rb

    def combine(self, y: torch.Tensor, off, mode, recv_topk_weights=None) -> tuple:
        out = torch.empty((self.R, self.T, self.H), dtype=torch.bfloat16, device="cuda")
        cw = (torch.empty((self.R, self.T, self.k), dtype=torch.float32, device="cuda")
              if recv_topk_weights is not None else None)
        ep.ep_combine(self.sh, y, off, self.lb.handle(), mode, self.topk, self.wts,
                      recv_topk_weights, out, cw, self.launch)
        return out, cw

    def ll_dispatch(self, use_fp8: bool, phase=ep.EP_PHASE_BOTH, buf: LLBuffers = None,
                    fp8_scale=ep.EP_FP8_SCALE_FP32, tensor_scale=0.0, packed=False) -> LLBuffers:
        buf = buf or LLBuffers(self.sh, use_fp8, fill=0x5A, fp8_scale=fp8_scale, tensor_scale=tensor_scale,
                               packed=packed)
        ep.ep_ll_dispatch(self.sh, self.x, self.topk, use_fp8, phase, buf.struct(), self.launch)
        return buf

    def ll_combine(self, y: torch.Tensor, buf: LLBuffers, phase=ep.EP_PHASE_BOTH) -> torch.Tensor:
        out = torch.empty((self.R, self.T, self.H), dtype=torch.bfloat16, device="cuda")
        ep.ep_ll_combine(self.sh, y, self.topk, self.wts, buf.struct(), phase, out, self.launch)
        return out
