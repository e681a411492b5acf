"""The seeded input generator: its whole-problem path against unit-by-unit generation."""


def test_generator_full_problem_equals_unit_by_unit_generation():
    """The input generator's one-run path (all sequences, all heads) gives exactly the values
    generating each sequence, or each head, on its own gives: the sampled parity tests
    regenerate single units and compare them with the full problem's outputs."""
    import torch
    from kda_gated_delta_04_gb300 import synth
    from kda_gated_delta_04_gb300.synth import PrefillWorkload
    for w in (PrefillWorkload("gen_check_bf16", 141, 3, 64, "bf16", (5, 0, 70, 1), 4, init_state=True),
              PrefillWorkload("gen_check_f32", 142, 2, 128, "f32", (130, 64), 2, init_state=True, raw_qk=True)):
        full = synth.prefill_inputs(w)
        cu = full["cu_seqlens"].tolist()
        for s in range(len(w.seq_lens)):
            one = synth.prefill_inputs(w, seqs=[s])
            for key in ("q", "k", "v", "log_alpha", "beta"):
                assert torch.equal(one[key], full[key][cu[s]:cu[s + 1]]), (w.name, s, key)
            assert torch.equal(one["init_state"][0], full["init_state"][s])
        for h in range(w.num_heads):
            one = synth.prefill_inputs(w, heads=[h])
            for key in ("q", "k", "v", "log_alpha"):
                assert torch.equal(one[key][:, 0], full[key][:, h]), (w.name, h, key)
            assert torch.equal(one["init_state"][:, 0], full["init_state"][:, h])
