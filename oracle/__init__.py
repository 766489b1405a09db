"""CPU oracle of the canvas-denoising core (test infrastructure only; see dgoracle)."""
