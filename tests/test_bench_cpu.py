"""Host-side pieces of bench.py (no GPU): where the roofline's measured DRAM
traffic comes from, and the attention parity bound."""
import glob
import os
import re

import numpy as np

import bench
import oracle
import synthetic_inputs as si

# kernel name in a profile's file name -> the source file it was captured from
KERNEL_SOURCE = {"tc_kernel": "tc.cu", "ffma_kernel": "ffma.cu", "skinny_kernel": "skinny.cu",
                 "gemv_kernel": "gemv.cu", "attn_fwd_kernel": "attn.cu", "bwd_ffma_kernel": "backward.cu"}


def _profiles_with_traffic():
    out = []
    for path in sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md"))):
        text = open(path).read()
        if "dram_bytes_per_launch:" not in text:
            continue
        base = os.path.basename(path)[:-3]
        kernel = next(k for k in KERNEL_SOURCE if base.startswith(k + "_"))
        out.append((kernel, base[len(kernel) + 1:], float(re.search(r"dram_bytes_per_launch:\s*([0-9.]+)", text)[1])))
    return out


def test_every_traffic_profile_matches_its_kernel_source():
    """A committed ncu summary feeds the bench's roofline `traffic` only while
    it was captured from the current kernel source: every summary that carries
    a per-launch DRAM figure must still match (recapture after a kernel
    change)."""
    profs = _profiles_with_traffic()
    assert len(profs) >= 15
    for kernel, workload, byts in profs:
        got = bench.traffic_from_profile(KERNEL_SOURCE[kernel], workload, kernel=kernel)
        assert got == byts, f"profiles/{kernel}_{workload}.md is stale against csrc/{KERNEL_SOURCE[kernel]}"


def test_traffic_is_null_for_a_changed_source(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "transformer_linear_layer_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    import hashlib

    sha = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles" / "k_kernel_w.md").write_text(
        f"dram_bytes_per_launch: 1234\n\nkernel_source_sha256_16: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("k.cu", "w") == 1234.0
    assert bench.traffic_from_profile("k.cu", "other") is None  # no summary for that workload
    (src / "k.cu").write_text("kernel v2\n")
    assert bench.traffic_from_profile("k.cu", "w") is None


def test_attention_bound_against_a_plain_loop():
    """bench.attention_bound = 1.05 * 2^-8 (sum_j p_ij |v_j| + |ref|) + 1e-5,
    checked against a loop over queries and keys on a tiny causal case."""
    att = si.Attention("tiny", 2, 5, 2, 64, causal=True, seed=3)
    qkv = si.make_qkv(att)
    scale = 0.125
    ref = oracle.attention(qkv, att.B, att.T, att.H, att.D, causal=True, scale=scale)
    got = bench.attention_bound(att, qkv, ref, scale)
    C, D = att.C, att.D
    want = np.zeros_like(ref)
    x = qkv.astype(np.float64)
    for b in range(att.B):
        for h in range(att.H):
            for i in range(att.T):
                qi = x[b * att.T + i, h * D:(h + 1) * D]
                s = [float(qi @ x[b * att.T + j, C + h * D:C + (h + 1) * D]) * scale for j in range(i + 1)]
                m = max(s)
                e = [np.exp(v - m) for v in s]
                tot = sum(e)
                a = sum(e[j] / tot * np.abs(x[b * att.T + j, 2 * C + h * D:2 * C + (h + 1) * D]) for j in range(i + 1))
                row = b * att.T + i
                want[row, h * D:(h + 1) * D] = 1.05 * 2.0 ** -8 * (a + np.abs(ref[row, h * D:(h + 1) * D])) + 1e-5
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)


def test_attention_workload_figures():
    att = si.GPT2_ATTN_B64
    assert att.algorithmic_bytes() == 50331648  # qkv read once (37.7 MB) and the output written once
    assert att.flops == 4 * 64 * 12 * (128 * 129 // 2) * 64
