"""CPU oracle package -- test infrastructure only (see ``oracle.sel_attn``)."""
