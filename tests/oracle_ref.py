"""Test helpers: run the oracle on (a sample of) a Case and compare with GPU results.

For large caches only the pages a sampled request touches are copied to the host; they
are re-packed into a compact page array with a remapped block table, so the oracle sees
exactly the same logical cache content.
"""
import numpy as np
import torch

import oracle

OUT_ATOL, OUT_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


def oracle_for(case, bs=None, hs=None, nthreads=0):
    """Oracle (out [b,h,512], lse [b,h]) for requests `bs` and heads `hs` of `case`."""
    B, H = case.B, case.H
    bs = list(range(B)) if bs is None else list(bs)
    hs = list(range(H)) if hs is None else list(hs)
    sl = case.seq_lens.cpu()
    bt = case.block_table.cpu()
    idx = case.indices.cpu() if case.indices is not None else None
    pages = []
    for b in bs:
        L = int(sl[b])
        if idx is None:
            n = (L + 63) // 64
            pages.append(bt[b, :n])
        else:
            lp = idx[b][idx[b] >= 0] // 64
            pages.append(bt[b, lp.unique()] if lp.numel() else bt[b, :0])
    used = torch.cat(pages).unique() if pages else torch.zeros(0, dtype=torch.int32)
    if used.numel() == 0:
        used = torch.zeros(1, dtype=torch.int32)
    lut = torch.zeros(case.num_pages, dtype=torch.int32)
    lut[used.long()] = torch.arange(used.numel(), dtype=torch.int32)
    compact = case.cache[used.to(case.cache.device).long()].cpu()
    bt_s = lut[bt[bs].long().clamp(0, case.num_pages - 1)].contiguous()
    qn = case.q_nope.cpu()[bs][:, hs].contiguous()
    qr = case.q_rope.cpu()[bs][:, hs].contiguous()
    sls = sl[bs].contiguous()
    if idx is not None:
        return oracle.decode_sparse(qn, qr, compact, bt_s, sls, idx[bs].contiguous(), case.scale,
                                    nthreads)
    if case.kv_dtype == "fp8":
        return oracle.decode_fp8(qn, qr, compact, bt_s, sls, case.scale, nthreads)
    return oracle.decode_dense(qn, qr, compact, bt_s, sls, case.scale, nthreads)


def assert_close(out, lse, ref_out, ref_lse, what=""):
    out = out.detach().cpu().double().numpy() if hasattr(out, "detach") else np.asarray(out)
    lse = lse.detach().cpu().double().numpy() if hasattr(lse, "detach") else np.asarray(lse)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    err = np.abs(out - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: out mismatch at {tuple(i)}: got {out[tuple(i)]} "
                             f"ref {ref_out[tuple(i)]} ({bad.sum()} of {bad.size} bad)")
    both_inf = np.isneginf(lse) & np.isneginf(ref_lse)
    lerr = np.where(both_inf, 0.0, np.abs(lse - ref_lse))
    badl = ~(lerr <= LSE_ATOL)
    if badl.any():
        i = np.argwhere(badl)[0]
        raise AssertionError(f"{what}: lse mismatch at {tuple(i)}: got {lse[tuple(i)]} "
                             f"ref {ref_lse[tuple(i)]}")


F16_UNIT = 2.0 ** -11   # unit roundoff of an fp16 operand (11 significant bits)


def fp8_operand_bound(case, b):
    """Largest score error the fp16 operands of the FP8-record decode can cause for request
    b, per head: the dequantised latent x = code x scale reaches the tensor core rounded to
    fp16 (|fp16(x) - x| <= 2^-11 |x|, plus 2^-25 below the normal range); the query is exact
    in fp16.  So |ds_t| <= scale * sum_c |q_c| (2^-11 |x_tc| + 2^-25), and the log-sum-exp
    of the scores moves by at most max_t |ds_t|."""
    import torch
    L = int(case.seq_lens[b])
    rec = case.cache
    bt = case.block_table.cpu()
    rows = torch.tensor([int(bt[b, t // 64]) * 64 + t % 64 for t in range(L)], dtype=torch.int64)
    flat = rec.reshape(-1, rec.shape[-1])[rows.to(rec.device)].cpu()
    codes = flat[:, :512].contiguous().view(torch.float8_e4m3fn).double()
    sc = flat[:, 512:528].contiguous().view(torch.float32).double()
    x = (codes * sc.repeat_interleave(128, dim=-1)).abs()                    # [L, 512]
    q = case.q_nope.cpu()[b].double().abs()                                 # [H, 512]
    return case.scale * (q @ (F16_UNIT * x + 2.0 ** -25).T).max(dim=1).values.numpy()


def assert_close_fp8(out, lse, ref_out, ref_lse, case, what=""):
    """FP8 records against the exact dequantisation: out within 1e-2 + 1e-2 |ref| everywhere;
    lse within 1e-3, or, for the (request, head) pairs where the fp16 rounding of the
    operands alone can move it by more, within 1e-3 plus that rounding's bound.  Returns
    the largest lse error seen."""
    out_np = out.detach().cpu().double().numpy() if hasattr(out, "detach") else np.asarray(out)
    lse_np = lse.detach().cpu().double().numpy() if hasattr(lse, "detach") else np.asarray(lse)
    err = np.abs(out_np - ref_out)
    bad = ~(err <= OUT_ATOL + OUT_RTOL * np.abs(ref_out))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: out mismatch at {tuple(i)}: got {out_np[tuple(i)]} ref {ref_out[tuple(i)]}")
    both_inf = np.isneginf(lse_np) & np.isneginf(ref_lse)
    lerr = np.where(both_inf, 0.0, np.abs(lse_np - ref_lse))
    for b in np.unique(np.argwhere(~(lerr <= LSE_ATOL))[:, 0]):
        bound = LSE_ATOL + fp8_operand_bound(case, int(b))
        if not np.all(lerr[b] <= bound):
            h = int(np.argmax(lerr[b] - bound))
            raise AssertionError(f"{what}: lse mismatch at ({b}, {h}): got {lse_np[b, h]} ref {ref_lse[b, h]}, "
                                 f"bound {bound[h]}")
    return float(np.nanmax(lerr)) if lerr.size else 0.0
