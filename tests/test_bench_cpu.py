"""Host-side pieces of bench.py: the source hash that keys the committed DRAM
traffic records (it ignores comment edits and notices code edits), and the
algorithmic FLOP and byte counts the roofline fractions divide by."""
import bench


def test_source_hash_ignores_comments_only():
    code = "int f(int a) {  // doubles\n    return 2 * a;\n}\n"
    recommented = "// header\nint f(int a) {  // twice a\n\n    return 2 * a;   \n}\n"
    edited = "int f(int a) {  // doubles\n    return 3 * a;\n}\n"
    assert bench.source_hash(code) == bench.source_hash(recommented)
    assert bench.source_hash(code) != bench.source_hash(edited)
    assert len(bench.source_hash(code)) == 16


def test_traffic_records_are_well_formed():
    # the records bench.py accepts for the current GEMM source (those whose
    # hash matches it) carry positive traffic above the weights' bytes
    recs = bench.traffic_record("gemm_tcgen05.cu")
    assert recs is not None
    for r in recs:
        assert r["dram_bytes_per_launch"] > r.get("weight_bytes", 0)


def test_algorithmic_work_of_the_default_workload():
    """The roofline denominators: the Mixtral-shaped layer at T = 16384 keeps
    all 32768 (token, slot) rows on 8 active experts."""
    import moe_inputs as mi

    w = mi.workload("mixtral")
    d, F, E, T, R = 4096, 14336, 8, 16384, 32768
    flops, bytes_, up_flops, up_bytes = bench.algorithmic(w, T, R, E)
    # up projection: two d x F products (W1, W3) per kept row
    assert up_flops == 2 * d * F * R * 2
    # its bytes: W1 and W3 of the active experts, the rows in, h out (bf16)
    assert up_bytes == 2 * d * F * 2 * E + R * d * 2 + R * F * 2 == 3087007744
    # layer: router (2 d E per token) and three d x F products per kept row
    assert flops == 2 * d * E * T + 2 * 3 * d * F * R
    # weights of the active experts, W_r in fp32, x in and y out (bf16)
    assert bytes_ == 3 * d * F * 2 * E + 4 * d * E + 2 * T * d * 2


def test_algorithmic_work_relu_and_shared_expert():
    import moe_inputs as mi

    sw = mi.workload("switch")                # ReLU: one d x F product up, one down
    f, _, uf, _ = bench.algorithmic(sw, 8192, 7000, 8)
    assert uf == 2 * 1024 * 4096 * 7000
    assert f == 2 * 1024 * 8 * 8192 + 2 * 2 * 1024 * 4096 * 7000
    ds = mi.workload("deepseek")              # shared expert: 6 d Fs per token
    f, b, _, _ = bench.algorithmic(ds, 128, 1024, 200)
    assert f == 2 * 7168 * 256 * 128 + 2 * 3 * 7168 * 2048 * 1024 + 6 * 7168 * 2048 * 128
    assert b == (3 * 7168 * 2048 * 2 * 200 + 3 * 7168 * 2048 * 2 + 4 * 7168 * 256
                 + 2 * 128 * 7168 * 2)
