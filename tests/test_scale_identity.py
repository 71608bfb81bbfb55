"""The quantizer computes the NVFP4 element factor e = fl(s_enc / E4M3(S)) of
"Add an NVFP4 quantization converter" (outer FP32 scale, inner E4M3 1x16
scale) without a division per block: every positive finite E4M3 value is
n * 2^j with n in 1..15, so e = fl(fl(s_enc / n) * 2^-j).  This checks that
identity in IEEE fp32 for every positive E4M3 code and tensor scales from the
smallest possible (2688 / FLT_MAX) to the overflow clamp (FLT_MAX), including
the overflow-to-infinity cases, on the CPU."""
import numpy as np

F32 = np.float32
FLT_MAX = np.finfo(np.float32).max


def e4m3_value(code: int) -> float:
    ex, man = code >> 3, code & 7
    if ex == 0:
        return man * 2.0 ** -9
    return (8 + man) * 2.0 ** (ex - 10)


def table_form(s_enc: np.float32, code: int) -> np.float32:
    ex, man = code >> 3, code & 7
    n = 8 + man if ex else man
    ex1 = ex if ex else 1
    q_n = F32(s_enc) / F32(n)                       # fl(s_enc / n)
    with np.errstate(over="ignore"):
        return F32(q_n * F32(2.0 ** (10 - ex1)))    # exact power-of-two scaling


def test_table_form_equals_division():
    rng = np.random.default_rng(5)
    amaxes = np.concatenate([
        np.array([FLT_MAX, FLT_MAX / 2, 3e38, 1e38, 1.0, 448.0, 6.0, 1e-3, 1e-30, 1e-37, 1.2e-38, 1e-40, 1e-45],
                 dtype=np.float32),
        (10.0 ** rng.uniform(-44, 38, 4000)).astype(np.float32),
    ])
    checked = 0
    for A in amaxes:
        with np.errstate(over="ignore", divide="ignore"):
            s_enc = F32(2688.0) / F32(A)
        if np.isinf(s_enc):
            s_enc = F32(FLT_MAX)      # the reading's overflow clamp
        for code in range(1, 0x7F):  # positive finite codes (0x7F is NaN)
            d = F32(e4m3_value(code))
            with np.errstate(over="ignore"):
                ref = F32(s_enc / d)
            got = table_form(s_enc, code)
            assert (np.isinf(ref) and np.isinf(got)) or ref == got, (A, code, ref, got)
            if not np.isinf(ref):
                assert ref >= np.finfo(np.float32).tiny  # e never subnormal
            checked += 1
    assert checked == len(amaxes) * 126
