"""CPU oracle for the paged LATENT attention operator (test infrastructure
only; the product path never imports it)."""
