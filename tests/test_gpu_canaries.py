"""Out-of-bounds writes, checked without a sanitizer: every buffer the library
writes (caches, mask, output, next slot(s), scores) sits between guard regions
filled with a sentinel, on shapes with ragged tails, and the guards must be
untouched after each entry point runs."""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf

import _pins
from _gpu import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side


def guarded(t: torch.Tensor, fill):
    """A copy of `t` inside a larger buffer; returns (view, whole buffer)."""
    n = t.numel()
    buf = torch.empty(n + 2 * GUARD, dtype=t.dtype, device="cuda")
    if t.dtype == torch.bfloat16:
        buf.view(torch.int16).fill_(fill)
    else:
        buf.fill_(fill)
    view = buf[GUARD:GUARD + n].view(t.shape)
    view.copy_(t)
    return view, buf


def guards_intact(buf, fill):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    if g.dtype == torch.bfloat16:
        return bool((g.view(torch.int16) == fill).all())
    return bool((g == fill).all())


@pytest.mark.parametrize("entry", ["step", "scores", "ex_topk", "attention", "noalloc"])
@pytest.mark.parametrize("d,g,S", [(64, 2, 77), (128, 4, 1000), (128, 8, 130)])
def test_no_write_outside_the_buffers(entry, d, g, S):
    rng = np.random.default_rng(d * 7 + g + S)
    Hkv = 2
    case = _pins.rand_case(rng, 3, Hkv * g, Hkv, d, S, p_masked=0.2, max_age=3 * S, ws_mode="any")
    B, Hq = 3, Hkv * g
    fill_bf, fill_i, fill_f = 0x1357, -777, -12345.5
    dev = {k: to_dev(v) for k, v in case.items()}
    k, kb = guarded(dev["k_cache"], fill_bf)
    v, vb = guarded(dev["v_cache"], fill_bf)
    mask, mb = guarded(dev["mask"], fill_i)
    out, ob = guarded(torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda"), fill_bf)
    kk = 7
    nxt_shape = (B, Hkv, kk) if entry == "ex_topk" else (B, Hkv)
    nxt, nb = guarded(torch.zeros(nxt_shape, dtype=torch.int32, device="cuda"), fill_i)
    scores, sb = guarded(torch.zeros(B, Hkv, S, dtype=torch.float32, device="cuda"), fill_f)
    args = (dev["q"], k, v, mask, dev["new_k"], dev["new_v"], dev["write_slot"])
    if entry == "step":
        lf.decode_step(*args, out, nxt, 4, 0.1)
    elif entry == "scores":
        lf.decode_step_scores(*args, out, nxt, scores, 4, 0.1)
    elif entry == "ex_topk":
        lf.decode_step_ex(*args, out, nxt, 4, 0.1, k=kk,
                          flags=lf.LF_STEP_FILL_EMPTY_FIRST | lf.LF_STEP_MASK_EVICTED,
                          scores=scores)
    elif entry == "attention":
        lf.decode_attention(*args, out, 0.1)
    else:
        lf.decode_step_noalloc(*args, out, nxt, 4, 0.1)
    torch.cuda.synchronize()
    for name, buf, fill in (("k_cache", kb, fill_bf), ("v_cache", vb, fill_bf), ("mask", mb, fill_i),
                            ("out", ob, fill_bf), ("next_slot", nb, fill_i), ("scores", sb, fill_f)):
        assert guards_intact(buf, fill), f"{entry}: write outside {name}"
    assert lf.device_errors() == 0
