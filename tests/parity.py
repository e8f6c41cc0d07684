"""Helpers for the GPU-vs-oracle parity tests.

The bar (restated from the operation's specification): forward O max abs error
<= 1e-2 and LSE abs error <= 1e-3; dQ, dK, dV relative L2 error <= 2e-2 each.
O and LSE are compared with the oracle whose rotated q', k' are the bf16
operands a tensor core consumes (oracle mode 1); gradients are compared with
the pure double oracle (mode 0).  O is judged on the kernel's fp32 output (the
same kernel rounds it to bf16 for the bf16 entry point; a separate check
requires the bf16 output to be exactly that rounding).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_TOL = 2e-2


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def packed_view(inp):
    """(q, k, v, dout) as [N, H, D] CPU tensors and the cu_seqlens list."""
    if "cu_seqlens" in inp:
        cu = [int(c) for c in inp["cu_seqlens"]]
        return [inp[n] for n in ("q", "k", "v", "dout")], cu
    B, T = inp["B"], inp["T"]
    H, D = inp["H"], inp["D"]
    ts = [inp[n].reshape(B * T, H, D) for n in ("q", "k", "v", "dout")]
    return ts, [i * T for i in range(B + 1)]


def run_gpu(inp, device="cuda", bwd=True, train=False):
    """Run the library on ``inp``; returns CPU tensors in the packed layout
    ([N, H, D] and LSE [H, N]).  ``train``: the bf16 forward and the backward
    are the training pair (rotated operands kept from forward to backward)."""
    from causal_self_attention_gb300 import ne_attn as na

    q, k, v, do = (inp[n].to(device) for n in ("q", "k", "v", "dout"))
    base, scale = inp["rope_base"], inp["scale"]
    res = {}
    if "cu_seqlens" in inp:
        cu = inp["cu_seqlens"].to(device)
        mx = inp["max_seqlen"]
        o32, lse = na.ne_attn_varlen_fwd(q, k, v, cu, mx, base, scale, out_f32=True)
        if train:
            o16, lse16, qr, kr = na.ne_attn_varlen_fwd_train(q, k, v, cu, mx, base, scale)
            if bwd:
                dq, dk, dv = na.ne_attn_varlen_bwd_train(qr, kr, v, o16, do, lse16, cu, mx, base,
                                                         scale)
        else:
            o16, lse16 = na.ne_attn_varlen_fwd(q, k, v, cu, mx, base, scale)
            if bwd:
                dq, dk, dv = na.ne_attn_varlen_bwd(q, k, v, o16, do, lse16, cu, mx, base, scale)
        res["lse"] = lse.cpu()
        res["lse_bf16call"] = lse16.cpu()
    else:
        o32, lse = na.ne_attn_fwd(q, k, v, base, scale, out_f32=True)
        if train:
            o16, lse16, qr, kr = na.ne_attn_fwd_train(q, k, v, base, scale)
            if bwd:
                dq, dk, dv = na.ne_attn_bwd_train(qr, kr, v, o16, do, lse16, base, scale)
        else:
            o16, lse16 = na.ne_attn_fwd(q, k, v, base, scale)
            if bwd:
                dq, dk, dv = na.ne_attn_bwd(q, k, v, o16, do, lse16, base, scale)
        B, H, T = lse.shape
        res["lse"] = lse.permute(1, 0, 2).reshape(H, B * T).cpu()
        res["lse_bf16call"] = lse16.permute(1, 0, 2).reshape(H, B * T).cpu()
    status = na.ne_attn_get_device_status()
    assert status == 0, f"device status {status} (code {na.ne_attn_last_device_code():#x})"
    H, D = inp["H"], inp["D"]
    res["o32"] = o32.reshape(-1, H, D).cpu()
    res["o16"] = o16.reshape(-1, H, D).cpu()
    if bwd:
        res.update(dq=dq.reshape(-1, H, D).cpu(), dk=dk.reshape(-1, H, D).cpu(),
                   dv=dv.reshape(-1, H, D).cpu())
    return res


def check_full(inp, gpu, bwd=True):
    """Compare every output with the full oracle.  Returns the error summary."""
    (q, k, v, do), cu = packed_view(inp)
    base, scale = inp["rope_base"], inp["scale"]
    ref1 = oracle.attention(q, k, v, None, cu, base=base, scale=scale, mode=1)
    errs = {}
    o32 = gpu["o32"].double().numpy()
    errs["o_max_abs"] = float(np.max(np.abs(o32 - ref1["o"])))
    errs["lse_max_abs"] = float(np.max(np.abs(gpu["lse"].double().numpy() - ref1["lse"])))
    # The bf16 entry point is the same kernel with the output rounded to bf16.
    assert torch.equal(gpu["o16"], gpu["o32"].to(torch.bfloat16)), "bf16 O != rne(fp32 O)"
    assert torch.equal(gpu["lse"], gpu["lse_bf16call"]), "LSE differs between out dtypes"
    assert errs["o_max_abs"] <= O_TOL, errs
    assert errs["lse_max_abs"] <= LSE_TOL, errs
    if bwd:
        ref0 = oracle.attention(q, k, v, do, cu, base=base, scale=scale, mode=0)
        for name in ("dq", "dk", "dv"):
            got = gpu[name].double().numpy()
            if np.linalg.norm(ref0[name]) == 0.0:
                # Every sequence has one row: its only softmax weight is 1, so
                # O = V and D = dO . O equals dP exactly, and dS, hence dQ and
                # dK, are exactly zero.  The kernels form dP - D from two fp32
                # sums of the same 64 exact products, in different orders: the
                # rounding residue is measured against the scale of dV.
                errs[name + "_rel_l2"] = float(np.linalg.norm(got) /
                                               max(np.linalg.norm(ref0["dv"]), 1e-300))
            else:
                errs[name + "_rel_l2"] = rel_l2(got, ref0[name])
        for name in ("dq", "dk", "dv"):
            assert errs[name + "_rel_l2"] <= GRAD_TOL, errs
    return errs


def check_sampled(inp, gpu, picks, bwd=True, long_loop_tiles=None):
    """Compare sampled rows with the oracle, for workloads too large for the
    full oracle.  ``picks``: list of (seq, head, qrows, krows).  O and LSE are
    checked row by row against the bound; gradients by relative L2 over the
    sampled rows.  With ``long_loop_tiles`` = n, the key rows whose gradients
    sum over at least n query tiles of 128 rows are also judged on their own
    (``dk_long_rel_l2``, ``dv_long_rel_l2``)."""
    (q, k, v, do), cu = packed_view(inp)
    base, scale = inp["rope_base"], inp["scale"]
    r1 = oracle.attention_sampled(q, k, v, None, cu, [(s, h, qr, []) for s, h, qr, _ in picks],
                                  base=base, scale=scale, mode=1)
    r0 = (oracle.attention_sampled(q, k, v, do, cu, picks, base=base, scale=scale, mode=0)
          if bwd else None)
    o_err = lse_err = 0.0
    acc = {n: ([], []) for n in ("dq", "dk", "dv", "dk_long", "dv_long")}
    for idx, (s, h, qrows, krows) in enumerate(picks):
        t0 = cu[s]
        qi = np.asarray(qrows) + t0
        o_err = max(o_err, float(np.max(np.abs(gpu["o32"][qi, h].double().numpy() - r1[idx]["o"]))))
        lse_err = max(lse_err, float(np.max(np.abs(gpu["lse"][h, qi].double().numpy() -
                                                    r1[idx]["lse"]))))
        if bwd:
            ki = np.asarray(krows) + t0
            acc["dq"][0].append(gpu["dq"][qi, h].double().numpy())
            acc["dq"][1].append(r0[idx]["dq"])
            if len(krows):
                acc["dk"][0].append(gpu["dk"][ki, h].double().numpy())
                acc["dk"][1].append(r0[idx]["dk"])
                acc["dv"][0].append(gpu["dv"][ki, h].double().numpy())
                acc["dv"][1].append(r0[idx]["dv"])
                if long_loop_tiles:
                    L = cu[s + 1] - cu[s]
                    sel = (L - np.asarray(krows)) > 128 * (long_loop_tiles - 1)
                    if sel.any():
                        for n in ("dk", "dv"):
                            acc[n + "_long"][0].append(gpu[n][ki[sel], h].double().numpy())
                            acc[n + "_long"][1].append(r0[idx][n][sel])
    errs = {"o_max_abs": o_err, "lse_max_abs": lse_err}
    assert torch.equal(gpu["o16"], gpu["o32"].to(torch.bfloat16)), "bf16 O != rne(fp32 O)"
    assert o_err <= O_TOL and lse_err <= LSE_TOL, errs
    if bwd:
        for n, (g, r) in acc.items():
            if g:
                errs[n + "_rel_l2"] = rel_l2(np.concatenate(g), np.concatenate(r))
                assert errs[n + "_rel_l2"] <= GRAD_TOL, errs
    return errs
