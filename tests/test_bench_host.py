"""Host-side pieces of the benchmark: the code hash that keys the committed ncu
traffic record, and the workload config both arms report."""
from __future__ import annotations

import bench


def test_code_hash_ignores_comments_only():
    src = "int f(int a) {\n  // the sum\n  return a + 1; /* one */\n}\n"
    edited_comment = "int f(int a) {\n  // the sum, plus one\n\n  return a + 1; /* 1 */\n}\n"
    edited_code = "int f(int a) {\n  // the sum\n  return a + 2; /* one */\n}\n"
    assert bench.code_text(src) == bench.code_text(edited_comment)
    assert bench.code_text(src) != bench.code_text(edited_code)
    files = {n: src for n in bench.KERNEL_SOURCES}
    h = bench.source_hash(lambda n: files[n])
    files[bench.KERNEL_SOURCES[0]] = edited_comment
    assert bench.source_hash(lambda n: files[n]) == h
    files[bench.KERNEL_SOURCES[0]] = edited_code
    assert bench.source_hash(lambda n: files[n]) != h


def test_both_arms_report_the_same_config():
    c = bench.residual_config(1)
    assert c["T"] == 32768 and c["D"] == 4096 and c["workload"] == "rmsnorm_residual fwd+bwd"
    assert bench.residual_config(4)["parallelism"] == "replicas x4"


def test_algorithmic_bytes_count_each_tensor_once():
    """The roofline numerators, rebuilt from the tensors each kernel must move
    once: bf16 activations of 2 bytes, an fp32 rstd of 4 bytes per row (w and
    dgamma, [D] each, are left out as negligible)."""
    T, D = 32768, 4096
    act, rstd = 2 * D, 4
    fwd = (act) + (act + act + rstd)                   # x in; y, x_copy, rstd out
    bwd = (act + act + act + rstd) + (act)             # g, x, g_res, rstd in; dx out
    assert bench.fwd_bytes(T, D) == T * fwd
    assert bench.bwd_pass1_bytes(T, D) == T * bwd
    assert bench.step_bytes(T, D) == T * (fwd + bwd) == 1_879_310_336


def test_ulp_histogram_of_the_bench_accuracy_sample():
    """The bench's accuracy sample counts each output's distance from the
    oracle's correctly rounded value in bf16 ulps: 0, 1, further but inside the
    cancellation clause, beyond."""
    import numpy as np
    ref = np.array([1.0, 1.0, -3.0, 0.0078125, 1.0, 1.0])
    ulp = bench._bf16_ulp(ref)
    assert ulp[0] == 2.0**-7 and ulp[2] == 2.0**-6 and ulp[3] == 2.0**-14
    got = ref + np.array([0.0, 1.0, -1.0, 0.0, 2.0, 3.0]) * ulp
    h = bench._ulp_histogram(got, ref)
    assert h == {"0": 2, "1": 2, "beyond": 2}
    pre = got.copy()                               # the unrounded value next to what the GPU returned
    scale = np.array([0.0, 0.0, 0.0, 0.0, 0.0, 1e-12])
    h = bench._ulp_histogram(got, ref, pre, scale)
    assert h == {"0": 2, "1": 2, "cancellation": 2, "beyond": 0}
    h = bench._ulp_histogram(got, ref, ref, scale)  # unrounded = the reference: 2 and 3 ulp are not cancellation
    assert h == {"0": 2, "1": 2, "cancellation": 0, "beyond": 2}
