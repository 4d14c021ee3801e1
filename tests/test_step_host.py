"""Host-side planning of KFACStep (no GPU): the layer groups that the
factor pass and the running-average pass overlap over."""
import pytest

import synth
from infra_fac_factors_gb300.step import LayerSpec, layer_groups


def specs(key):
    cfg = synth.config(key)
    return [LayerSpec(l.d_in, l.d_out, cfg.rows(l), cfg.batch, l.hw) for l in cfg.layers]


@pytest.mark.parametrize("key", ["single_linear", "mlp", "resnet_conv", "bert_layer", "bert_large"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 200])
def test_layer_groups_partition_in_order(key, n):
    layers = specs(key)
    groups = layer_groups(layers, n)
    assert 1 <= len(groups) <= min(n, len(layers))
    assert groups[0][0] == 0 and groups[-1][1] == len(layers)
    for (b0, e0), (b1, e1) in zip(groups, groups[1:]):
        assert e0 == b1
    assert all(e > b for b, e in groups)


def test_layer_groups_balance_bert_large():
    layers = specs("bert_large")
    groups = layer_groups(layers, 4)
    assert len(groups) == 4
    work = [sum(L.rows * L.d_in ** 2 + L.rows * L.d_out ** 2 for L in layers[b:e]) for b, e in groups]
    assert max(work) <= 1.1 * min(work)
