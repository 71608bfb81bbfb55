"""The quantizer's stochastic-rounding arithmetic (index-domain form: three
round-up lines, a minimum, and a magic-number ceiling that also carries the
sign) makes the same decision as the rounding rule of "Add an NVFP4
quantization converter" ("What changed": Philox-keyed, unbiased stochastic
rounding, read as r < ceil(2^16 frac)).  The probe restates both in C with the
directed roundings emulated exactly and compares them on every finite bf16
value, a strided fp32 sweep, random pairs and all 2^16 draws around every grid
point; no GPU is needed."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_index_domain_sr_equals_the_rounding_rule(tmp_path):
    exe = str(tmp_path / "sr_index_domain")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", os.path.join(HERE, "probes", "sr_index_domain.c"), "-o", exe,
                    "-lm"], check=True)
    r = subprocess.run([exe, "20000000"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
    assert "mismatches 0" in r.stdout
