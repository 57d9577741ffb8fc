"""Reads the plan bytes written by the library's planner (host twin or device)."""
import numpy as np


def _up(x, a=256):
    return (x + a - 1) // a * a


def parse(buf, B, H):
    buf = np.asarray(buf, dtype=np.uint8)
    hd = buf[:64].view(np.int32)
    magic, b_, h_, topk, units, n_items, max_items, max_partials, per, n_part = [int(v) for v in hd[:10]]
    assert magic == 0x4D4C4150 and b_ == B and h_ == H
    o = 256
    ub = buf[o:o + 4 * (units + 1)].view(np.int32).copy()
    o = _up(o + 4 * (units + 1))
    items = buf[o:o + 16 * max_items].view(np.int32).reshape(max_items, 4)[:n_items].copy()
    o = _up(o + 16 * max_items)
    ns = buf[o:o + 4 * B].view(np.int32).copy()
    o = _up(o + 4 * B)
    sb = buf[o:o + 4 * B].view(np.int32).copy()
    o = _up(o + 4 * B)
    rs = buf[o:o + 8 * B].view(np.int64).copy()
    o = _up(o + 8 * B)
    iu = buf[o:o + 4 * max_items].view(np.int32)[:n_items].copy()
    o = _up(o + 4 * max_items)
    n_split = int(hd[10])
    sl = buf[o:o + 4 * B].view(np.int32)[:n_split].copy()
    o = _up(o + 4 * B)
    return dict(req_start=rs, item_unit=iu, topk=topk, units=units, n_items=n_items, max_items=max_items,
                max_partials=max_partials, per=per, n_partials=n_part, unit_begin=ub,
                items=items, num_splits=ns, split_base=sb, split_list=sl, n_split_reqs=n_split,
                plan_end=o)
