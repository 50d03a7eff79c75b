"""The Python binding checks every tensor of a call against q and k before
anything reaches the library: the C ABI sees only pointers and sizes, so a
mismatched shape, dtype or LSE size would let a kernel read or write past a
caller's buffer.  Shapes are checked before the device, so CPU tensors reach
these checks; a well-formed CPU call then fails on the device check (there is
no CPU path)."""

import pytest
import torch

from tiled_attention_07_gb300 import fa

BF = torch.bfloat16


def t(*shape, dtype=BF):
    return torch.zeros(*shape, dtype=dtype)


def fwd_args(B=1, H=2, Nq=128, Nk=256, d=64):
    return dict(q=t(B, H, Nq, d), k=t(B, H, Nk, d), v=t(B, H, Nk, d), o=t(B, H, Nq, d),
                lse=torch.zeros(B, H, Nq))


def call_fwd(a):
    fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], 0.125, False)


def test_well_formed_cpu_call_fails_on_the_device_only():
    with pytest.raises(ValueError, match="CUDA tensors only"):
        call_fwd(fwd_args())


@pytest.mark.parametrize("name,bad,err,match", [
    ("k", t(1, 2, 256, 80), ValueError, "k has shape"),        # head dim differs from q
    ("k", t(1, 3, 256, 64), ValueError, "k has shape"),        # head count differs
    ("k", t(256, 2, 64), ValueError, "k has shape"),           # 3-D beside a 4-D q
    ("v", t(1, 2, 200, 64), ValueError, "v has shape"),        # fewer keys than k
    ("o", t(1, 2, 127, 64), ValueError, "o has shape"),        # one row short
    ("v", t(1, 2, 256, 64, dtype=torch.float16), TypeError, "v is torch.float16"),
    ("k", t(1, 2, 256, 64, dtype=torch.float16), TypeError, "k is torch.float16"),
    ("lse", torch.zeros(1, 2, 100), ValueError, "lse must be"),
    ("lse", torch.zeros(1, 2, 128, dtype=torch.float64), ValueError, "lse must be"),
    ("lse", torch.zeros(1, 2, 256)[..., ::2], ValueError, "lse must be"),   # not contiguous
])
def test_fwd_mismatch_is_rejected(name, bad, err, match):
    a = fwd_args()
    a[name] = bad
    with pytest.raises(err, match=match):
        call_fwd(a)


def test_seq_heads_d_layout_passes_the_shape_checks():
    a = dict(q=t(128, 2, 64), k=t(300, 2, 64), v=t(300, 2, 64), o=t(128, 2, 64), lse=torch.zeros(2, 128))
    with pytest.raises(ValueError, match="CUDA tensors only"):
        call_fwd(a)


def bwd_args(B=1, H=2, Nq=128, Nk=256, d=64):
    a = fwd_args(B, H, Nq, Nk, d)
    a.update(do=t(B, H, Nq, d), dq=t(B, H, Nq, d), dk=t(B, H, Nk, d), dv=t(B, H, Nk, d))
    return a


def call_bwd(a, fn="fa_bwd"):
    args = [a[n] for n in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv")]
    if fn == "fa_bwd":
        fa.fa_bwd(*args, 0.125, True)
    elif fn == "fa_bwd_noalloc":
        fa.fa_bwd_noalloc(*args, 0.125, True)
    else:
        fa.fa_bwd_phase(fa.FA_BWD_DKDV, *args, 0.125, True, t(1 << 16, dtype=torch.uint8))


@pytest.mark.parametrize("fn", ["fa_bwd", "fa_bwd_noalloc", "fa_bwd_phase"])
@pytest.mark.parametrize("name,bad,match", [
    ("do", t(1, 2, 256, 64), "do has shape"),     # dO shaped like K
    ("dq", t(1, 2, 120, 64), "dq has shape"),
    ("dk", t(1, 2, 128, 64), "dk has shape"),     # dK shaped like Q
    ("dv", t(1, 2, 256, 80), "dv has shape"),
    ("lse", torch.zeros(1, 2, 64), "lse must be"),
])
def test_bwd_mismatch_is_rejected(fn, name, bad, match):
    a = bwd_args()
    a[name] = bad
    with pytest.raises(ValueError, match=match):
        call_bwd(a, fn)


@pytest.mark.parametrize("fn", ["fa_bwd", "fa_bwd_noalloc", "fa_bwd_phase"])
def test_bwd_well_formed_cpu_call_fails_on_the_device_only(fn):
    with pytest.raises(ValueError, match="CUDA tensors only"):
        call_bwd(bwd_args(), fn)


def test_bwd_gradient_dtype_must_match():
    a = bwd_args()
    a["dv"] = t(1, 2, 256, 64, dtype=torch.float16)
    with pytest.raises(TypeError, match="dv is torch.float16"):
        call_bwd(a)


def test_split_and_fp8v_check_shapes():
    a = fwd_args()
    a["o"] = t(1, 2, 100, 64)
    with pytest.raises(ValueError, match="o has shape"):
        fa.fa_fwd_split(a["q"], a["k"], a["v"], a["o"], a["lse"], 0.125, False, 2)
    a = fwd_args()
    vt = torch.zeros(1, 2, 64, 256, dtype=torch.uint8)
    a["lse"] = torch.zeros(1, 2, 64)
    with pytest.raises(ValueError, match="lse must be"):
        fa.fa_fwd_fp8v(a["q"], a["k"], vt, a["o"], a["lse"], 0.125, False)
    with pytest.raises(ValueError, match="vt must be"):
        fa.fa_fwd_fp8v(a["q"], a["k"], vt[..., :200], a["o"], torch.zeros(1, 2, 128), 0.125, False)


def test_softmax_shape_check_precedes_the_device_check():
    with pytest.raises(ValueError, match="same shape"):
        fa.fa_softmax_rows(torch.zeros(4, 100), torch.zeros(4, 99))
    with pytest.raises(ValueError, match="CUDA tensors only"):
        fa.fa_softmax_rows(torch.zeros(4, 100), torch.zeros(4, 100))
