"""The fp32-scale quotient of the CUDA kernels (correctly rounded reciprocal,
one FMA residual correction -- Markstein's method -- run two at a time on
negated operands) equals IEEE division on every (x, scale) pair the cast can
produce, except where the true quotient is below 2^-64 (the residual
underflows there); in those cases both values encode to the same signed zero
(CPU only, exhaustive over about 1.07e9 pairs per format).

IEEE fp32 multiply, FMA and division round identically on the host and the
GPU (no flush to zero on either side), so the host enumeration proves the
device arithmetic.  The CUDA source is checked to still use that sequence
(the packed negated-operand form, in every kernel that divides by an fp32
scale).

The power-of-two scales' exponent is taken from the bits of the floored
amax instead of dividing; that rule is checked against the definition
(exponent of RN(max(a, 1e-4) / fmt_max), rounded up to a power of two) for
every positive finite fp32 amax of both formats.
"""
import os
import platform
import re
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "quotient_check.c")
EXP_SRC = os.path.join(HERE, "pow2_exponent_check.c")
CU = os.path.join(ROOT, "precision_quantization_token_gb300", "csrc",
                  "tk_device.cuh")


def _has_fma_flag():
    try:
        return " fma " in open("/proc/cpuinfo").read().replace("\n", " ")
    except OSError:
        return False


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("q") / "quotient_check")
    flags = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math"]
    if platform.machine() in ("x86_64", "AMD64") and _has_fma_flag():
        flags.append("-mfma")          # hardware fused multiply-add for fmaf
    subprocess.run(["gcc", *flags, "-o", exe, SRC, "-lm"], check=True)
    return exe


@pytest.fixture(scope="module")
def results(checker):
    """Both formats' enumerations, run as two processes at once."""
    procs = {f: subprocess.Popen([checker, f], stdout=subprocess.PIPE,
                                 stderr=subprocess.PIPE, text=True)
             for f in ("448", "6")}
    out = {}
    for f, p in procs.items():
        stdout, stderr = p.communicate(timeout=900)
        assert p.returncode == 0, stderr
        out[f] = (stdout, stderr)
    return out


def test_kernels_use_the_correctly_rounded_reciprocal():
    """inv = RN(1/s): the IEEE reciprocal of the fp32 ratio, in group_scale."""
    src = open(CU).read()
    assert re.search(r"g\.inv = __frcp_rn\(r\);", src)


def test_packed_kernels_use_the_negated_form():
    """quotient2 (fp32 scales): nx = -x from the sign-flipped BF16 pair;
    q0 = nx*ninv; r = fma(q0, s, nx); q = fma(r, ninv, q0), with ninv the
    negated reciprocal (quotient2_inv) -- the form the checker compares."""
    src = open(CU).read()
    body = src[src.index("__device__ __forceinline__ void quotient2("):]
    body = body[body.index("} else {"):body.index("\n}\n")]
    seq = re.findall(r'"(xor\.b32|mul\.rn\.f32x2|fma\.rn\.f32x2) ([^;]*);', body)
    assert seq == [("xor.b32", "n, %2, 0x80008000"),
                   ("mul.rn.f32x2", "q0, nx, %4"),
                   ("fma.rn.f32x2", "r, q0, %3, nx"),
                   ("fma.rn.f32x2", "q, r, %4, q0")], seq
    assert '"r"(w), "l"(s2), "l"(inv2)' in body
    inv = src[src.index("float quotient2_inv("):]
    assert "return POW2 ? g.inv : -g.inv;" in inv[:200]


def test_fp32_input_paths_use_the_negated_form():
    """The SwiGLU and RMSNorm casts run the same negated-operand sequence
    on values they form negated (-y), with the negated reciprocal."""
    src = open(os.path.join(os.path.dirname(CU), "tk_cast.cu")).read()
    sw = src[src.index("__device__ __forceinline__ void cast_chunk("):]
    sw = sw[:sw.index("\n}\n")]
    assert "const uint64_t ni = pack_f32x2(-gs.inv, -gs.inv);" in sw
    assert "const uint64_t q0 = fmul2(ny[i], ni);" in sw
    assert "r = ffma2(ffma2(q0, s2, ny[i]), ni, q0);" in sw
    # both SwiGLU paths form -y directly: the packed fast path with the
    # denominator negated, RN(t * -1 + -1), the per-element path through
    # swiglu_neg (the same scalar sequence, or -(the IEEE fallback))
    assert "const uint64_t d = ffma2(pack_f32x2(t0, t1), m1, m1);" in sw
    assert "ny[i] = pack_f32x2(swiglu_neg(" in sw
    neg = src[src.index("float swiglu_fast_neg(float gate, float up) {"):]
    neg = neg[:neg.index("\n}\n")]
    assert '"f"(-1.0f - t)' in neg and "return (gate * up) * r;" in neg
    assert ": -swiglu_ieee(gate, up);" in src
    rms = src[src.index("__device__ __forceinline__ void rms_chunk("):]
    rms = rms[:rms.index("\n}\n")]
    assert "const float f = POW2 ? rstd : -rstd;" in rms      # -y for fp32 scales
    assert "const float iv = quotient2_inv<POW2>(gs);" in rms
    assert "const uint64_t q0 = fmul2(y2[i], i2);" in rms
    assert "r = ffma2(ffma2(q0, s2, y2[i]), i2, q0);" in rms


@pytest.mark.parametrize("fmt_max", ["448", "6"])
def test_every_reachable_pair(results, fmt_max):
    stdout, stderr = results[fmt_max]
    pairs, bad, sub, sub_bad, form = map(int, stdout.split())
    assert pairs > 10 ** 9
    assert bad == 0, stderr
    assert sub_bad == 0
    assert form == 0, "the negated-operand form differs from the sequence"
    print(f"{pairs} pairs; {sub} quotients below 2^-64 off by the residual "
          "underflow, all encoding to the same signed zero")


@pytest.fixture(scope="module")
def exponent_results(tmp_path_factory):
    """The exponent rule over every positive finite fp32 amax, for both
    formats, and the wrong rule (mantissa field >= the threshold) that the
    enumeration must reject; four processes at once."""
    exe = str(tmp_path_factory.mktemp("e") / "pow2_exponent_check")
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off",
                    "-fno-fast-math", "-o", exe, EXP_SRC], check=True)
    runs = {(f, m): subprocess.Popen([exe, f, *([m] if m else [])],
                                     stdout=subprocess.PIPE,
                                     stderr=subprocess.PIPE, text=True)
            for f in ("448", "6") for m in ("", "ge")}
    out = {}
    for key, p in runs.items():
        stdout, stderr = p.communicate(timeout=900)
        assert p.returncode == 0, stderr
        out[key] = tuple(map(int, stdout.split())) + (stderr,)
    return out


def test_kernels_take_the_exponent_from_the_amax_bits():
    """group_scale's power-of-two branch: e = E - 8 (E4M3) or E - 2 (E2M1),
    plus one when the mantissa field exceeds 1.75's (0x600000) or 1.5's
    (0x400000); the fp32 branch keeps the IEEE division."""
    src = open(CU).read()
    body = src[src.index("GroupScale group_scale(float amax) {"):]
    body = body[:body.index("\n}\n")]
    assert "kDrop = FMT == TK_FMT_E4M3 ? 8u : 2u;" in body
    assert "kMant = FMT == TK_FMT_E4M3 ? 0x600000u : 0x400000u;" in body
    assert "const float a = fmaxf(amax, 1e-4f);" in body
    assert "g.e = (u >> 23) - kDrop + ((u & 0x7FFFFFu) > kMant);" in body
    assert "const float r = __fdiv_rn(a, kMax);" in body


@pytest.mark.parametrize("fmt_max", ["448", "6"])
def test_exponent_rule_on_every_amax(exponent_results, fmt_max):
    values, bad, stderr = exponent_results[(fmt_max, "")]
    assert values == 0x7F800000          # +0 through the largest finite fp32
    assert bad == 0, stderr
    # the enumeration does tell rules apart: >= in place of > must fail
    wrong_values, wrong_bad, _ = exponent_results[(fmt_max, "ge")]
    assert wrong_values == values and wrong_bad > 0
