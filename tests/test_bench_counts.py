"""bench.py's launch-count claim (`gpu_launches`) against the launch lists
captured with ncu on the same workloads: eight library kernels per e8_swiglu
forward step (router 2: weight split and the fused logits/softmax/top-k
kernel, whose last CTA writes the probability sums; dispatch histograms +
ranks + row scatter 3; up and down GEMMs; combine with the aux loss) and 20
per training step (23 for e128_top8_T32768); two more router kernels above 64 experts (the finishing
kernel and the probability sums); one more dispatch kernel (the
per-expert scan of the chunk histograms) above 65536 assignments; one more for
the global aux loss of token-sharded replicas."""
import argparse
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _args(**over):
    a = dict(gather=False, z_beta=None, train=False)
    a.update(over)
    return argparse.Namespace(**a)


def test_forward_and_training_launch_counts(monkeypatch):
    b = _bench()
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    e8 = b.synth.workload("e8_swiglu")
    assert b.KERNELS_PER_STEP_TOTAL(e8, _args()) == 8
    assert b.KERNELS_PER_STEP_TOTAL(e8, _args(train=True)) == 20
    assert b.KERNELS_PER_STEP_TOTAL(e8, _args(gather=True)) == 7          # no row scatter
    assert b.KERNELS_PER_STEP_TOTAL(e8, _args(z_beta=1e-3)) == 9         # + z-loss
    e64 = b.synth.workload("e64_zipf")
    assert b.KERNELS_PER_STEP_TOTAL(e64, _args()) == 8
    e128 = b.synth.workload("e128_top8_T32768")       # E > 64: + finishing kernel; T*k > 65536: + chunk scan
    assert b.KERNELS_PER_STEP_TOTAL(e128, _args()) == 11
    assert b.KERNELS_PER_STEP_TOTAL(e128, _args(train=True)) == 23   # the e128 training launch list
    monkeypatch.setenv("WORLD_SIZE", "2")                                  # replicas: + global aux loss
    assert b.KERNELS_PER_STEP_TOTAL(e8, _args()) == 9
