"""Host-side logic of bench.py that needs no GPU: how a layer's linears are grouped into
bd_linear_batch calls, and the reference arm's stand-in library."""
import bench


def test_layer_groups_follow_the_projections_that_share_an_input():
    names = ["L0.q", "L0.k", "L0.v", "L0.o", "L0.gate", "L0.up", "L0.down",
             "L1.q", "L1.k", "L1.v", "L1.o", "L1.gate", "L1.up", "L1.down"]
    assert bench.layer_groups(names) == [[0, 1, 2], [3], [4, 5], [6], [7, 8, 9], [10], [11, 12], [13]]


def test_layer_groups_never_cross_layers_or_join_unrelated_matrices():
    assert bench.layer_groups(["L0.v", "L1.q", "L1.k"]) == [[0], [1, 2]]
    assert bench.layer_groups(["L0.up", "L0.gate"]) == [[0, 1]]
    assert bench.layer_groups(["L0.attn_sq", "L0.mlp_up", "L0.mlp_down"]) == [[0], [1], [2]]
    assert bench.layer_groups([]) == []


def test_reference_stand_in_answers_the_workload_constructors():
    lib = bench._NoLib()
    assert lib.bd_compress_batch_workspace_size(None) > 0
    assert lib.bd_linear_batch_workspace_size(None) > 0
    assert lib.linear_descs([1, 2]) == [1, 2]
    try:
        lib.bd_linear(None)
    except RuntimeError:
        pass
    else:
        raise AssertionError("the stand-in must refuse GPU calls")
