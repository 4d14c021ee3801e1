"""Host logic of bench.py that needs no GPU: the one-GPU rule, the kernel
tables, the committed-traffic lookup and the oracle leg's layer sample."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run_bench(args, env_extra=None):
    # the refusal must come before any GPU work: the child reports whether
    # torch (and with it CUDA) was ever imported
    code = ("import sys, runpy; sys.argv = ['bench.py'] + %r\n"
            "try:\n    runpy.run_path('bench.py', run_name='__main__')\n"
            "except SystemExit as e:\n    print('torch' in sys.modules, file=sys.stderr); raise\n") % (args,)
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=120)


@pytest.mark.parametrize("args,env", [(["--gpus", "2"], None), (["--gpus", "8", "--impl", "reference"], None),
                                      ([], {"WORLD_SIZE": "2"}), (["--gpus", "0"], None)])
def test_bench_refuses_anything_but_one_gpu_before_gpu_work(args, env):
    r = _run_bench(args, env)
    assert r.returncode == 2, r.stderr
    assert "refused" in r.stderr
    assert r.stderr.strip().splitlines()[-1] == "False"  # torch never imported
    assert r.stdout == ""


def test_one_gpu_is_accepted():
    args = bench.parse([])
    assert args.gpus == 1
    assert bench.multi_gpu_refusal(args, {}) is None
    assert bench.multi_gpu_refusal(args, {"WORLD_SIZE": "1"}) is None
    assert bench.multi_gpu_refusal(args, {"WORLD_SIZE": "4"}) is not None
    assert bench.multi_gpu_refusal(bench.parse(["--gpus", "2"]), {}) is not None


def test_bench_tables_cover_every_profiled_kernel_kind():
    # the bench reads every kind of the library's launch profile: each needs a
    # kernel name for the roofline line, its source file and, if tensor-bound,
    # its MMA count
    from infra_fac_factors_gb300 import capi

    assert set(bench.KERNEL_NAMES) == set(capi.KERNEL_KINDS)
    assert set(bench.KERNEL_SOURCES) == set(capi.KERNEL_KINDS)
    assert set(bench.ISSUED_PER_ALGORITHMIC) == set(capi.KERNEL_KINDS) - {"running"} - set(bench.CUDA_CORE_KINDS)
    for name in bench.KERNEL_SOURCES.values():
        assert len(bench.source_digest(name)) == 12


def test_traffic_figure_only_while_the_kernel_source_is_unchanged(tmp_path):
    dig = bench.source_digest("inverse_tc.cu")
    p = tmp_path / "traffic.md"
    p.write_text("# summary\n"
                 f"`traffic inv_update bert_large 123456789 {dig}`\n"
                 "traffic inv_lauum bert_large 5 000000000000\n")
    assert bench.traffic_figure("inv_update", "bert_large", str(p)) == 123456789.0
    assert bench.traffic_figure("inv_update", "bert_layer", str(p)) is None
    assert bench.traffic_figure("inv_lauum", "bert_large", str(p)) is None  # stale digest
    assert bench.traffic_figure("inv_update", "bert_large", str(tmp_path / "none.md")) is None


def test_committed_traffic_lines_are_well_formed():
    if not os.path.exists(bench.TRAFFIC_FILE):
        pytest.skip("no committed traffic figures")
    with open(bench.TRAFFIC_FILE) as f:
        lines = [l.strip().strip("`").split() for l in f if l.strip().strip("`").startswith("traffic ")]
    for parts in lines:
        assert len(parts) == 5 and parts[1] in bench.KERNEL_SOURCES and float(parts[3]) > 0


def test_oracle_sample_covers_every_layer_but_the_stack():
    import synth

    for key in ("single_linear", "mlp", "resnet_conv", "bert_layer"):
        cfg = synth.config(key)
        ids, scale = bench.oracle_layer_sample(cfg, "auto")
        assert ids == list(range(len(cfg.layers))) and scale == 1.0
    big = synth.config("bert_large")
    ids, scale = bench.oracle_layer_sample(big, "auto")
    assert ids == [0, 1, 2, 3] and scale == 24.0
    # the sample is one encoder layer: its four shapes repeat in every other one
    shapes = [(l.d_in, l.d_out) for l in big.layers]
    assert all(shapes[i] == shapes[i % 4] for i in range(len(shapes)))
    assert bench.oracle_layer_sample(big, "all") == (list(range(96)), 1.0)


def test_reference_arm_prints_one_line_for_one_gpu(capsys):
    args = bench.parse(["--impl", "reference", "--config", "single_linear", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
